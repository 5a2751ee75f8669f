// qs_fused.cu -- the whole decode-sized MoE-FFN layer in one persistent kernel (sm_103a).
//
// One CTA per SM (its shared memory admits no second one), every CTA resident at
// once.  The kernel is a programmatic dependent launch: the next call in the
// stream is launched while this one still runs, and its CTAs take each SM as
// soon as this call's CTA there leaves.  Before it waits for the previous grid
// (griddepcontrol.wait) the producer warp only prefetches weights into L2; no
// thread touches x, the workspace or the output before that wait.  A CTA has
// one producer warp and 15 consumer warps.  The producer streams the CTA's
// routing-independent tiles from HBM into a ring of 21 KB shared-memory stages
// with bulk asynchronous copies (TMA engine): one "full" mbarrier per stage
// counts the bytes in, one "empty" mbarrier per stage tells the producer the
// stage may be refilled.  Tiles, in the order every CTA walks them (tile i of
// the grid belongs to CTA i mod gridDim):
//
//   router rows (fp32)  |  shared gate/up rows (bf16)  |  [routed gate/up rows (Q2_K)]  |  [down groups]
//
// (For one token, or a ring of fewer than three stages, group B reads the shared gate/up
// rows from global memory instead, prefetched into L2 at the start.)
// The routed gate/up rows and the down groups (RD output rows: the shared
// expert's bf16 down rows and every active expert's Q2_K down rows) are
// numbered as tiles but do not pass through the ring: the warps that use them
// load them from global memory into registers, after the CTA's warps have
// requested all of the routed rows into L2 at once (the shared expert's down
// rows are prefetched at the start).  One SM's copy engine works through its
// copies one after another, and a down group of many experts would be many
// copies of a few hundred bytes held in stages while long tasks run; the load
// path keeps far more of them in flight.
// Consumers work as independent warp tasks, so different warps can be in
// different phases at once and nothing waits on a CTA-wide barrier:
//   group A (warps 0-7):  router rows -> logits; then the routing
//                         (top-k, softmax, grouping of the T*k entries by expert)
//   group B (warps 8-14): x scales, int16 x and sigmoid gates; shared gate/up rows -> hs
//   then every warp, round robin over the CTA's remaining tasks:
//     routed gate/up rows -> h;  staging of hs and of each entry's int16 h;
//     down rows: shared-expert down row + every active expert's down row -> out,
//     summed in a fixed order (ascending expert id, then the gated shared expert)
//
// Cross-CTA exchange: logits, hs and h are plain fp32 arrays in the workspace,
// each with a 64-bit completion counter in the workspace header.  A CTA that
// has written its share of an array (all of its rows of that kind, possibly
// none) adds 1 to the counter with one release reduction; one thread per CTA
// waits with acquire loads until the counter reaches this call's target, and
// only then does the CTA read the array, once.  (Readers that poll the data
// words themselves keep the lines being written under a stream of loads, and
// on this part that delays the writes by microseconds.)  The counters are never
// reset: every call adds exactly gridDim to each of them and to the exit
// counter (a CTA that winds down early adds what it has not added yet when it
// leaves), so call n's target is (n + 1) * gridDim, n being the exit count the
// call finds when it starts divided by gridDim.  Every wait is bounded by the
// global timer; a wait that runs out sets the sticky status QS_ERR_TIMEOUT and
// the CTA winds down.
#include "qs_common.cuh"
#include "qs_internal.h"
#include "qs_q2k.cuh"
#include "qs_fmt.cuh"
#include "qs_warp.cuh"

#include <algorithm>

namespace qs {

// 16 warps at one CTA per SM leave 128 registers per thread (a seventeenth warp would put five
// warps on one of the SM's four schedulers and cap every thread at 96)
constexpr int kCW = 15;                  // consumer warps
constexpr int kCT = kCW * 32;            // consumer threads
constexpr int kGWA = 8;                  // warps of consumer group A (router rows, routing)
constexpr int kGWB = kCW - kGWA;         // warps of consumer group B (x preparation, shared gate/up rows)
constexpr int kGTA = kGWA * 32;
constexpr int kGTB = kGWB * 32;
constexpr int kFusedThreads = kCT + 32;  // + the producer warp
constexpr int kStageBytes = 21504;       // 2 x 128 Q2_K row-blocks of 84 B
constexpr int kMaxStages = 12;
constexpr int kMaxEnt = 128;             // T * k
constexpr int kMaxT = kFusedMaxT;
constexpr int kMaxCand = 512;            // tokens x 32-logit chunks x min(k, 32) this kernel takes; larger
                                         // calls (12-16 tokens of 256 experts) ran faster on the tensor cores
constexpr int kMaxRD = 16;

struct FusedParams {
    const void* x;
    const float* Wr;
    const float* bias;
    const uint8_t* experts;
    int64_t stride;
    const uint16_t* sg;
    const uint16_t* su;
    const uint16_t* sd;
    const uint16_t* ssig;
    float* out;
    float* xlog;  // [T x E] logits
    float* xhs;   // [T x S] hs
    float* xh;    // [T*k x F] h, rows in sorted entry order
    WsHeader* hdr;
    int32_t* rec_ids;  // [T*k] the call's routing (written by CTA 0)
    float* rec_p;      // [T*k]
    int H, E, k, F, S, T, x_dtype;
    int RR, RS, R, RD;  // rows per router, shared gate/up, routed gate/up and down tile
    int nstages;
    int x_sys;  // x is host memory reached through its mapped address: the consumer warps load it
    int sg_direct;  // group B reads the shared gate/up rows from global memory (no shared tiles in the ring)
    // byte offsets inside the data region that follows FusedCtl
    int off_xq, off_sig, off_hsf, off_hq, off_pbuf, off_stages;
};

struct alignas(16) FusedCtl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t xbar;  // x and w_sg
    // one-shot events inside the CTA, waited on with the waiters suspended in hardware
    uint64_t routed_bar;  // the routing is published
    uint64_t xq_bar;      // x scales, int16 x and gates are staged
    uint64_t shared_bar;  // group B has finished its shared gate/up rows (x and w_sg are free)
    uint64_t hs_bar;      // hs is staged
    uint64_t h_bar;       // every CTA's h is published
    uint64_t staged_bar;  // every entry's int16 h is staged (T * k arrivals)
    int done[kMaxStages];  // tasks finished on the tile now in each stage
    int slot_seq[kMaxStages];  // sequence number of the tile a stage is being filled with
    int abort, issued, n_active, pad1;
    int et_left;   // routed gate/up tasks of this CTA not finished yet
    int h_poller;  // set by the one warp that waits for the h counter
    int published; // bit i: this CTA has added its 1 to exchange counter i (kPubLogits, kPubHs, kPubH)
    uint64_t target;  // this call's target of every exchange counter
    int ids[kMaxEnt];
    float p[kMaxEnt];
    int ent_sorted[kMaxEnt];     // entries t*k+slot sorted by (expert, entry)
    int es[kMaxEnt];             // expert of ent_sorted[i]
    int es_tok[kMaxEnt];         // token of ent_sorted[i]
    int act_e[kMaxEnt];          // active experts, ascending
    const uint8_t* act_w[kMaxEnt];  // first byte of each active expert's weights
    int act_begin[kMaxEnt + 1];  // first ent_sorted index of each active expert
    int tok_sorted[kMaxEnt];     // per token, its k ent_sorted indices, ascending
    int wcnt[8];
    float gate_s[kMaxT];
    float xscale[kMaxT];
    float hscale[kMaxEnt];       // scale of the int16 h row of ent_sorted[i]
    float ps[kMaxEnt];           // routing weight of ent_sorted[i]
    float red[2 * kGTB];
};

// Named barriers of the consumer groups: 2 for group A, 3 for group B.
template <int NT>
__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(NT) : "memory"); }

// number of threads of consumer group `id` whose predicate is true (a group barrier of NT threads)
template <int NT>
__device__ __forceinline__ int group_count(int id, bool pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %2, 0;\n\t"
        "bar.red.popc.u32 %0, %1, %3, p;\n\t}"
        : "=r"(r)
        : "r"(id), "r"((int)pred), "n"(NT)
        : "memory");
    return r;
}

// One thread: wait with acquire loads until the exchange counter *c reaches `target`.
// False if the CTA is aborting or the wait outlasts kWaitNs.
__device__ __forceinline__ bool wait_count(const uint64_t* c, uint64_t target, const int* abort) {
    if (ld_acquire_u64(c) >= target) return true;
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_u64(c) < target) {
        if (*reinterpret_cast<const volatile int*>(abort) || global_timer_ns() - t0 > kWaitNs) return false;
    }
    return true;
}

enum { kPubLogits = 1, kPubHs = 2, kPubH = 4 };

// One thread: add this CTA's 1 to an exchange counter (release: the CTA's rows of that kind,
// ordered before this thread by a barrier or a fence, become visible first).
__device__ __forceinline__ void publish(FusedCtl& C, uint64_t* ctr, int bit) {
    red_release_add_u64(ctr, 1);
    atomicOr(&C.published, bit);
}

// ------------------------------------------------------------------ tile and task bookkeeping

struct Plan {
    int G, cta;
    int n_rt, n_st, n_ind;    // router tiles, shared gate/up tiles, routing-independent total
    int tpe;                  // routed gate/up tiles per active expert
    int n_dg;                 // down groups
    int rowH, rowF;           // Q2_K row bytes along H and along F
    int own_rt, own_st;       // tiles of each kind this CTA owns
    int cpr, rpw, ept;        // Q2_K chunks per gate/up row, rows per task, tasks per tile
    int cpf, epp;             // chunks per down row, experts per warp pass
};

__device__ __forceinline__ int first_owned(int lo, int G, int cta) {
    const int r = lo % G;
    return lo + ((cta - r) % G + G) % G;
}
__device__ __forceinline__ int owned_count(int lo, int hi, int G, int cta) {
    const int f = first_owned(lo, G, cta);
    return f < hi ? (hi - 1 - f) / G + 1 : 0;
}

// n / d and n % d for 0 <= n < 2^24 through a float reciprocal and one correction step
// (cheaper than an integer division by a value known only at run time).
struct FDiv {
    float inv;
    int d;
};
__device__ __forceinline__ FDiv fdiv_of(int d) { return FDiv{1.0f / (float)d, d}; }
__device__ __forceinline__ int fdiv(int n, const FDiv& f, int& rem) {
    int q = __float2int_rz(__int2float_rn(n) * f.inv);
    int r = n - q * f.d;
    if (r < 0) {
        q--;
        r += f.d;
    } else if (r >= f.d) {
        q++;
        r -= f.d;
    }
    rem = r;
    return q;
}

__device__ __forceinline__ Plan make_plan(const FusedParams& P, int block_bytes) {
    Plan L;
    L.G = gridDim.x;
    L.cta = blockIdx.x;
    L.n_rt = P.E / P.RR;
    L.n_st = P.S > 0 ? P.S / P.RS : 0;
    L.n_ind = L.n_rt + L.n_st;
    L.tpe = P.F / P.R;
    L.n_dg = P.H / P.RD;
    L.rowH = P.H / kBlockWeights * block_bytes;
    L.rowF = P.F / kBlockWeights * block_bytes;
    L.own_rt = owned_count(0, L.n_rt, L.G, L.cta);
    L.own_st = owned_count(L.n_rt, L.n_ind, L.G, L.cta);
    L.cpr = 4 * (P.H / kBlockWeights);
    L.rpw = L.cpr >= 32 ? 1 : 32 / L.cpr;
    L.ept = P.R / L.rpw;
    L.cpf = 4 * (P.F / kBlockWeights);
    L.epp = 32 / L.cpf;
    return L;
}

// ------------------------------------------------------------------ waits (bounded, warp-uniform outcome)

// Whole warp waits for an mbarrier phase; false if any lane gave up or the CTA is aborting.
__device__ __forceinline__ bool warp_wait_bar(FusedCtl& C, uint64_t* bar, uint32_t parity) {
    const bool ok = !vload(&C.abort) && mbar_wait(bar, parity);
    return __all_sync(0xffffffffu, ok);
}

// Whole warp waits for tile `seq` in its stage.  A warp may run laps ahead of the
// producer, so it first waits until the stage is being filled with this very
// tile (parity alone cannot tell laps apart), then for the stage's bytes.
__device__ __forceinline__ bool warp_wait_tile(FusedCtl& C, int seq, int ns) {
    const int slot = seq % ns;
    bool ok = true;
    if (vload(&C.slot_seq[slot]) != seq) {
        const uint64_t t0 = global_timer_ns();
        while (vload(&C.slot_seq[slot]) != seq) {
            if (vload(&C.abort) || global_timer_ns() - t0 > kWaitNs) {
                ok = false;
                break;
            }
            __nanosleep(32);
        }
    }
    ok = ok && !vload(&C.abort) && mbar_wait(&C.full[slot], (seq / ns) & 1);
    return __all_sync(0xffffffffu, ok);
}

// Whole warp waits for an mbarrier phase, suspended in hardware between polls (each poll
// wakes at the latest after 1 us to look at the abort flag); false on abort or time-out.
__device__ __forceinline__ bool warp_wait_mbar(FusedCtl& C, uint64_t* bar, uint32_t parity) {
    bool ok = true;
    if (!mbar_try_wait(bar, parity)) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait_sleep(bar, parity, 1000)) {
            if (vload(&C.abort) || global_timer_ns() - t0 > kWaitNs) {
                ok = false;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok && !vload(&C.abort));
}

__device__ __forceinline__ void fail(FusedCtl& C, uint32_t* status) {
    if ((threadIdx.x & 31) == 0) {
        set_status(status, QS_ERR_TIMEOUT);
        vstore(&C.abort, 1);
    }
}

// A task is done with the tile in stage `slot` (ntask tasks share it): the last
// one hands the stage back to the producer.
__device__ __forceinline__ void release_slot(FusedCtl& C, int slot, int ntask) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        if (atomicAdd(&C.done[slot], 1) == ntask - 1) {
            C.done[slot] = 0;
            mbar_arrive(&C.empty[slot]);
        }
    }
}

// ------------------------------------------------------------------ producer warp

// lane 0 waits until stage seq % ns is free (bounded), then marks it as holding
// tile seq; outcome broadcast to the warp
__device__ __forceinline__ bool producer_slot(FusedCtl& C, int seq, int ns) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        if (seq >= ns) {
            ok = (!vload(&C.abort) && mbar_wait(&C.empty[seq % ns], (seq / ns - 1) & 1)) ? 1 : 0;
            if (!ok) vstore(&C.abort, 1);
        }
        if (ok) vstore(&C.slot_seq[seq % ns], seq);
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ void producer(const FusedParams& P, FusedCtl& C, uint8_t* data) {
    const Plan L = make_plan(P, kBlockBytes);  // the tile counts only (no routed row sizes)
    const int lane = threadIdx.x & 31;
    const int ns = P.nstages;
    uint8_t* stages = data + P.off_stages;
    int seq = 0;
    auto slot = [&](int s) { return stages + (size_t)(s % ns) * kStageBytes; };
    auto bar = [&](int s) { return &C.full[s % ns]; };

    // weights first, into L2 only (the previous kernel in the stream may still be running and
    // an L2 prefetch cannot make a later read stale), then wait for that kernel to complete
#pragma unroll 1
    for (int g = L.cta + lane * L.G; g < L.n_ind; g += 32 * L.G) {
        if (g < L.n_rt) {
            const uint32_t bytes = (uint32_t)P.RR * P.H * 4;
            bulk_prefetch_l2(P.Wr + (size_t)g * P.RR * P.H, bytes);
        } else {
            const int j = g - L.n_rt;
            const uint32_t bytes = (uint32_t)P.RS * P.H * 2;
            bulk_prefetch_l2(P.sg + (size_t)j * P.RS * P.H, bytes);
            bulk_prefetch_l2(P.su + (size_t)j * P.RS * P.H, bytes);
        }
    }
    // the shared expert's down rows do not depend on the routing either: one slice per CTA
    if (P.S > 0) {
#pragma unroll 1
        for (int r = L.cta + lane * L.G; r < P.H; r += 32 * L.G)
            bulk_prefetch_l2(P.sd + (size_t)r * P.S, (uint32_t)P.S * 2);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // x and the shared-expert gate vector first: group A and group B start on them
    {
        const uint32_t xb = (uint32_t)P.T * P.H * (P.x_dtype == QS_BF16 ? 2 : 4);
        const uint32_t sb = P.S > 0 ? (uint32_t)P.H * 2 : 0u;
        if (lane == 0) mbar_arrive_expect_tx(&C.xbar, (P.x_sys ? 0u : xb) + sb);
        __syncwarp();
        if (lane == 0 && !P.x_sys) bulk_g2s(data, P.x, xb, &C.xbar);
        if (lane == 1 && sb) bulk_g2s(data + P.off_sig, P.ssig, sb, &C.xbar);
    }
    // router rows, then shared gate/up rows (unless group B reads those from global memory)
    const int n_tiles = P.sg_direct ? L.n_rt : L.n_ind;
#pragma unroll 1
    for (int g = L.cta; g < n_tiles; g += L.G) {
        if (!producer_slot(C, seq, ns)) goto done;
        if (g < L.n_rt) {
            const uint32_t bytes = (uint32_t)P.RR * P.H * 4;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(seq), bytes);
                fence_proxy_async_smem();
                bulk_g2s(slot(seq), P.Wr + (size_t)g * P.RR * P.H, bytes, bar(seq));
            }
        } else {
            const int j = g - L.n_rt;
            const uint32_t bytes = (uint32_t)P.RS * P.H * 2;
            if (lane == 0) mbar_arrive_expect_tx(bar(seq), 2 * bytes);
            __syncwarp();
            if (lane < 2) {
                fence_proxy_async_smem();
                bulk_g2s(slot(seq) + lane * bytes, (lane ? P.su : P.sg) + (size_t)j * P.RS * P.H, bytes, bar(seq));
            }
        }
        __syncwarp();
        seq++;
    }
done:
    if (lane == 0) vstore(&C.issued, seq);
}

// ------------------------------------------------------------------ warp-level arithmetic

// ------------------------------------------------------------------ the kernel

// FMT: the routed experts' weight format (kFmtQ2K, kFmtQ4K).
template <int MAXT, int FMT>
__global__ void __launch_bounds__(kFusedThreads, 1) fused_decode_kernel(const FusedParams P) {
    using FO = FmtOps<FMT>;
    extern __shared__ __align__(128) uint8_t smem[];
    FusedCtl& C = *reinterpret_cast<FusedCtl*>(smem);
    uint8_t* data = smem + (sizeof(FusedCtl) + 127) / 128 * 128;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = P.H, E = P.E, k = P.k, F = P.F, S = P.S, T = P.T;
    const int n_ent = T * k;
    const bool x_f32 = P.x_dtype != QS_BF16;
    uint32_t* status = &P.hdr->status;
    uint64_t* ctr_exit = reinterpret_cast<uint64_t*>(&P.hdr->ctr[kCtrExit][0]);
    uint64_t* ctr_lg = reinterpret_cast<uint64_t*>(&P.hdr->ctr[kCtrLogits][0]);
    uint64_t* ctr_hs = reinterpret_cast<uint64_t*>(&P.hdr->ctr[kCtrHs][0]);
    uint64_t* ctr_h = reinterpret_cast<uint64_t*>(&P.hdr->ctr[kCtrH][0]);
    const uint8_t* xraw = data;                                              // [T x H] as given
    uint32_t* xqf = reinterpret_cast<uint32_t*>(data + P.off_xq);            // [T][H/64 chunks][36] fragments
    const uint8_t* sigbuf = data + P.off_sig;                                // [H] bf16
    float* hsf = reinterpret_cast<float*>(data + P.off_hsf);                 // [T x S]
    uint32_t* hqf = reinterpret_cast<uint32_t*>(data + P.off_hq);            // [T*k][F/64 chunks][36] fragments
    float* pbuf = reinterpret_cast<float*>(data + P.off_pbuf);               // [consumer warps x kMaxEnt]
    uint8_t* stages = data + P.off_stages;
    const int ns = P.nstages;

    if (tid == 0) {
        for (int i = 0; i < ns; i++) {
            mbar_init(&C.full[i], 1);
            mbar_init(&C.empty[i], 1);
            C.done[i] = 0;
            C.slot_seq[i] = -1;
        }
        mbar_init(&C.xbar, 1);
        mbar_init(&C.routed_bar, 1);
        mbar_init(&C.xq_bar, 1);
        mbar_init(&C.shared_bar, 1);
        mbar_init(&C.hs_bar, 1);
        mbar_init(&C.h_bar, 1);
        mbar_init(&C.staged_bar, (uint32_t)(P.T * P.k));
        C.abort = C.issued = C.n_active = 0;
        C.et_left = C.h_poller = C.published = 0;
        C.target = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kCW) {
        producer(P, C, data);
    } else {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        // every earlier call has left (the wait above), none of this call can leave before this
        // CTA publishes its logits: the exit count is an exact multiple of gridDim here
        if (tid == 0) C.target = (ld_relaxed_u64(ctr_exit) / gridDim.x + 1) * gridDim.x;
        const Plan L = make_plan(P, FO::kBlock);
        const int gtid = warp < kGWA ? tid : tid - kGTA, gwarp = warp < kGWA ? warp : warp - kGWA;
        if (P.x_sys) {  // x from mapped host memory: every load in flight, then the stores
            const int nv = P.T * P.H * (x_f32 ? 4 : 2) / 16;
            const uint4* src = static_cast<const uint4*>(P.x);
            uint4* dst = reinterpret_cast<uint4*>(data);
#pragma unroll 1
            for (int i0 = tid; i0 < nv; i0 += 4 * kCT) {
                uint4 v[4];
#pragma unroll
                for (int z = 0; z < 4; z++)
                    if (i0 + z * kCT < nv) v[z] = __ldcv(src + i0 + z * kCT);
#pragma unroll
                for (int z = 0; z < 4; z++)
                    if (i0 + z * kCT < nv) dst[i0 + z * kCT] = v[z];
            }
            asm volatile("bar.sync 4, %0;" ::"n"(kCT) : "memory");  // every consumer warp
        }
        bool ok = warp_wait_bar(C, &C.xbar, 0);
        if (!ok) fail(C, status);

        if (warp < kGWA) {
            // ------------------------------------------------------ group A: router rows
#pragma unroll 1
            for (int idx = gwarp; ok && idx < L.own_rt * P.RR; idx += kGWA) {
                const int m = idx / P.RR, r = idx % P.RR;
                const int g = L.cta + m * L.G;
                if (!(ok = warp_wait_tile(C, m, ns))) break;
                float acc[MAXT];
                warp_dense_row<MAXT>(stages + (size_t)(m % ns) * kStageBytes + (size_t)r * H * 4, true, H, xraw, x_f32,
                                     T, acc);
                const int e = g * P.RR + r;
                const float b = P.bias ? P.bias[e] : 0.0f;
#pragma unroll
                for (int t = 0; t < MAXT; t++)
                    if (t < T && lane == t) P.xlog[(size_t)t * E + e] = acc[t] + b;
                release_slot(C, m % ns, P.RR);
            }
            if (!ok) fail(C, status);
            // ------------------------------------------------------ group A: routing
            // group-uniform outcome of the previous waits; the barrier also orders every
            // logit this group stored before the release below
            ok = group_count<kGTA>(2, !ok) == 0;
            if (ok) {
                bool got = true;
                if (gtid == 0) {
                    publish(C, ctr_lg, kPubLogits);
                    got = wait_count(ctr_lg, C.target, &C.abort);
                }
                ok = group_count<kGTA>(2, !got) == 0;
            }
            if (ok) {
                // top-k of each token's logits and the softmax over the k (one warp per token)
#pragma unroll 1
                for (int t = gwarp; t < T; t += kGWA) {
                    int id;
                    float w;
                    if (E <= 256) warp_topk<8>(P.xlog + (size_t)t * E, E, k, id, w);
                    else warp_topk_stream(P.xlog + (size_t)t * E, E, k, id, w);
                    if (lane < k) {
                        C.ids[t * k + lane] = id;
                        C.p[t * k + lane] = w;
                    }
                }
                group_sync<kGTA>(2);
                if (MAXT == 1 || n_ent <= 32) {  // (the one-token kernel runs only with k <= 32)
                    // one warp: entries ordered by (expert, entry) with shuffles, then the active
                    // experts and each token's entries, without further group barriers
                    if (gwarp == 0) {
                        const bool act = lane < n_ent;
                        const int e = act ? C.ids[lane] : 0x7fffffff;
                        int rank = 0;
#pragma unroll 1
                        for (int j = 0; j < n_ent; j++) {
                            const int f = __shfl_sync(0xffffffffu, e, j);
                            rank += (f < e) | ((f == e) & (j < lane));
                        }
                        if (act) {
                            C.ent_sorted[rank] = lane;
                            C.ps[rank] = C.p[lane];
                            C.es[rank] = e;
                            C.es_tok[rank] = lane / k;
                        }
                        __syncwarp();
                        // lane: sorted position
                        const int er = act ? C.es[lane] : -1;
                        const int eprev = __shfl_up_sync(0xffffffffu, er, 1);
                        const bool start = act && (lane == 0 || er != eprev);
                        const unsigned bal = __ballot_sync(0xffffffffu, start);
                        const int ai = __popc(bal & ((2u << lane) - 1u)) - 1;
                        if (start) {
                            C.act_e[ai] = er;
                            C.act_w[ai] = P.experts + (int64_t)er * P.stride;
                            C.act_begin[ai] = lane;
                        }
                        if (lane == n_ent - 1) {
                            C.act_begin[ai + 1] = n_ent;
                            C.n_active = ai + 1;
                        }
                        const int tr = act ? C.es_tok[lane] : -1;
                        const unsigned same = __match_any_sync(0xffffffffu, tr);
                        if (act) C.tok_sorted[tr * k + __popc(same & ((1u << lane) - 1u))] = lane;
                        if (blockIdx.x == 0 && act) {  // the call's routing, for the caller to read back
                            P.rec_ids[lane] = C.ids[lane];
                            P.rec_p[lane] = C.p[lane];
                        }
                        __syncwarp();
                        if (lane == 0) {
                            const int n_et = C.n_active * L.tpe;
                            C.et_left = owned_count(L.n_ind, L.n_ind + n_et, L.G, L.cta) * L.ept;
                            if (C.et_left == 0) publish(C, ctr_h, kPubH);  // no routed rows here
                            mbar_arrive(&C.routed_bar);
                        }
                    }
                } else {
                    // order the entries by (expert, entry)
#pragma unroll 1
                    for (int i = gtid; i < n_ent; i += kGTA) {
                        const int e = C.ids[i];
                        int rank = 0;
#pragma unroll 8
                        for (int j = 0; j < n_ent; j++) {
                            const int f = C.ids[j];
                            rank += (f < e) | ((f == e) & (j < i));
                        }
                        C.ent_sorted[rank] = i;
                        C.ps[rank] = C.p[i];
                        C.es[rank] = e;
                        C.es_tok[rank] = i / k;
                    }
                    group_sync<kGTA>(2);
                    // active experts: a run start in es[] opens a new active expert
                    const bool start = gtid < n_ent && (gtid == 0 || C.es[gtid] != C.es[gtid - 1]);
                    const unsigned bal = __ballot_sync(0xffffffffu, start);
                    if (lane == 0 && gwarp < 4) C.wcnt[gwarp] = __popc(bal);
                    group_sync<kGTA>(2);
                    if (gtid < n_ent) {
                        int a = __popc(bal & ((2u << lane) - 1u)) - 1;
#pragma unroll 1
                        for (int w = 0; w < gwarp; w++) a += C.wcnt[w];
                        if (start) {
                            C.act_e[a] = C.es[gtid];
                            C.act_w[a] = P.experts + (int64_t)C.es[gtid] * P.stride;
                            C.act_begin[a] = gtid;
                        }
                        if (gtid == n_ent - 1) {
                            C.act_begin[a + 1] = n_ent;
                            C.n_active = a + 1;
                        }
                        const int t = C.es_tok[gtid];
                        int pos = 0;
#pragma unroll 8
                        for (int j = 0; j < gtid; j++) pos += C.es_tok[j] == t;
                        C.tok_sorted[t * k + pos] = gtid;
                    }
                    if (blockIdx.x == 0) {  // the call's routing, for the caller to read back
                        for (int i = gtid; i < n_ent; i += kGTA) {
                            P.rec_ids[i] = C.ids[i];
                            P.rec_p[i] = C.p[i];
                        }
                    }
                    group_sync<kGTA>(2);
                    if (gtid == 0) {
                        const int n_et = C.n_active * L.tpe;
                        C.et_left = owned_count(L.n_ind, L.n_ind + n_et, L.G, L.cta) * L.ept;
                        if (C.et_left == 0) publish(C, ctr_h, kPubH);  // no routed rows here
                        mbar_arrive(&C.routed_bar);
                    }
                }
            } else {
                fail(C, status);
            }
        } else {
            // ------------------------------------------------------ group B: x scales, int16 x, gates
            ok = group_count<kGTB>(3, !ok) == 0;
            if (ok) {
                float mx[MAXT], gz[MAXT];
#pragma unroll
                for (int t = 0; t < MAXT; t++) mx[t] = gz[t] = 0.0f;
#pragma unroll 1
                for (int i = gtid * 8; i < H; i += kGTB * 8) {
                    float sv[8];
                    if (S > 0) load8(sigbuf + (size_t)i * 2, false, sv);
#pragma unroll
                    for (int t = 0; t < MAXT; t++) {
                        if (t < T) {
                            float xv[8];
                            load8(xraw + ((size_t)t * H + i) * (x_f32 ? 4 : 2), x_f32, xv);
#pragma unroll
                            for (int q = 0; q < 8; q++) {
                                mx[t] = fmaxf(mx[t], fabsf(xv[q]));
                                if (S > 0) gz[t] = fmaf(sv[q], xv[q], gz[t]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < MAXT; t++) {
                    if (t < T) {
                        const float m = warp_max(mx[t]);
                        const float z = warp_sum(gz[t]);
                        if (lane == 0) {
                            C.red[gwarp * MAXT + t] = m;
                            C.red[kGTB + gwarp * MAXT + t] = z;
                        }
                    }
                }
                group_sync<kGTB>(3);
                if (gtid < T) {
                    float m = 0.0f, z = 0.0f;
#pragma unroll 1
                    for (int w = 0; w < kGWB; w++) {
                        m = fmaxf(m, C.red[w * MAXT + gtid]);
                        z += C.red[kGTB + w * MAXT + gtid];
                    }
                    C.xscale[gtid] = m;
                    C.gate_s[gtid] = sigmoid(z);
                }
                group_sync<kGTB>(3);
                // int16 x in fragment layout; each 8-value group is one 16-byte store, the
                // two groups of a 16-value shift group are adjacent lanes (sums via shuffle)
#pragma unroll 1
                for (int i0 = gtid * 8; i0 < ((T * H + 255) / 256) * 256; i0 += kGTB * 8) {
                    const bool live = i0 < T * H;
                    const int t = live ? i0 / H : 0, p = live ? i0 - t * H : 0;
                    const float m = C.xscale[t];
                    const float inv = m > 0.0f ? 32767.0f / m : 0.0f;
                    float xv[8];
                    if (live) load8(xraw + (size_t)i0 * (x_f32 ? 4 : 2), x_f32, xv);
                    uint32_t wq[4];
                    int sum = 0;
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const int a0 = live ? __float2int_rn(xv[2 * q] * inv) : 0;
                        const int a1 = live ? __float2int_rn(xv[2 * q + 1] * inv) : 0;
                        wq[q] = (uint32_t)(a0 & 0xffff) | ((uint32_t)a1 << 16);
                        sum += a0 + a1;
                    }
                    FO::put8(xqf + (size_t)t * (H / 64) * kFragWords, p, wq, sum, live);
                }
                group_sync<kGTB>(3);
                if (gtid == 0) mbar_arrive(&C.xq_bar);
            } else {
                fail(C, status);
            }
            // ------------------------------------------------------ group B: shared gate/up rows
#pragma unroll 1
            for (int idx = gwarp; ok && idx < L.own_st * P.RS; idx += kGWB) {
                const int m = idx / P.RS, r = idx % P.RS;
                const int sq = L.own_rt + m;
                const int j = first_owned(L.n_rt, L.G, L.cta) + m * L.G - L.n_rt;
                const size_t row = (size_t)j * P.RS + r;
                const uint8_t *gw, *uw;
                if (MAXT == 1 || P.sg_direct) {  // from global memory (prefetched into L2 before the previous
                                                 // grid ended; always for one token)
                    gw = reinterpret_cast<const uint8_t*>(P.sg + row * H);
                    uw = reinterpret_cast<const uint8_t*>(P.su + row * H);
                } else {
                    if (!(ok = warp_wait_tile(C, sq, ns))) break;
                    const uint8_t* st = stages + (size_t)(sq % ns) * kStageBytes;
                    gw = st + (size_t)r * H * 2;
                    uw = st + (size_t)(P.RS + r) * H * 2;
                }
                float ga[MAXT], ua[MAXT];
                if (MAXT > 1) {  // several tokens: both rows in one pass over the activations
                    warp_dense_rows2<MAXT>(gw, uw, H, xraw, x_f32, T, ga, ua);
                } else {  // one token: one row at a time, four loads of each in flight
                    warp_dense_row<MAXT>(gw, false, H, xraw, x_f32, T, ga);
                    warp_dense_row<MAXT>(uw, false, H, xraw, x_f32, T, ua);
                }
#pragma unroll
                for (int t = 0; t < MAXT; t++)
                    if (t < T && lane == t) P.xhs[(size_t)t * S + row] = silu(ga[t]) * ua[t];
                if (!(MAXT == 1 || P.sg_direct)) release_slot(C, sq % ns, P.RS);
            }
            if (!ok) fail(C, status);
            // every hs row of this CTA is stored: publish them (the barrier orders the stores)
            if (group_count<kGTB>(3, !ok) == 0 && gtid == 0) {
                publish(C, ctr_hs, kPubHs);
                mbar_arrive(&C.shared_bar);
            }
        }

        // ---------------------------------------------------------- every warp: the routed part
        if (ok && !(ok = warp_wait_mbar(C, &C.routed_bar, 0))) fail(C, status);
        const int na = ok ? C.n_active : 0;
        const int n_et = na * L.tpe;
        const int own_et = owned_count(L.n_ind, L.n_ind + n_et, L.G, L.cta);
        const int lo_dg = L.n_ind + n_et;
        const int own_dg = owned_count(lo_dg, lo_dg + L.n_dg, L.G, L.cta);
        const int n_stage_tasks = (S > 0 ? 1 : 0) + n_ent;
        const int q_et = own_et * L.ept;              // pool: routed gate/up tasks
        const int q_all = q_et + n_stage_tasks + own_dg * P.RD;
        // ---------------------------------------------------------- routed gate/up rows
        // Tasks q = warp, warp + kCW, ... below q_et.  A lane owns chunk c0 + i * cstep (i < nch) of
        // row rl of the task; its chunks are one stream, loaded one item ahead of the one computed
        // (so the next task's rows are in flight while this task is reduced and stored).  Per entry
        // of the expert, the chunk dots are added in chunk order, then across lanes.
        int q = warp;
        if (ok && q < q_et) {
            if (!(ok = warp_wait_mbar(C, &C.xq_bar, 0))) fail(C, status);
        }
        const int rl = L.cpr >= 32 ? 0 : lane / L.cpr;
        const int c0 = L.cpr >= 32 ? lane : lane % L.cpr;
        const int cstep = L.cpr >= 32 ? 32 : L.cpr;
        const int nch = L.cpr / cstep;
        const unsigned gm = L.cpr >= 32 ? 0xffffffffu : (((1u << L.cpr) - 1u) << (lane & ~(L.cpr - 1)));
        const int g0 = first_owned(L.n_ind, L.G, L.cta);
        // A task's position: tile m of this CTA, task rt inside it, active expert a and its tile
        // tt.  Found by division once, then advanced by kCW tasks with a few subtractions.
        struct TaskPos {
            int rt, a, tt;
        };
        auto task_pos = [&](int qq) {
            TaskPos t;
            const int m = qq / L.ept;
            t.rt = qq - m * L.ept;
            const int idx = g0 + m * L.G - L.n_ind;
            t.a = idx / L.tpe;
            t.tt = idx - t.a * L.tpe;
            return t;
        };
        auto task_next = [&](TaskPos& t) {
            t.rt += kCW;
            while (t.rt >= L.ept) {  // next tile of this CTA: G tiles further
                t.rt -= L.ept;
                t.tt += L.G;
            }
            while (t.tt >= L.tpe) {
                t.tt -= L.tpe;
                t.a++;
            }
        };
        // first byte of this lane's gate row of a task (the up row is F rows further)
        auto task_row = [&](const TaskPos& t) -> const uint8_t* {
            return C.act_w[t.a] + (int64_t)(t.tt * P.R + t.rt * L.rpw + rl) * L.rowH;
        };
        const int64_t up_off = (int64_t)P.F * L.rowH;
        // one token and one chunk per lane: that chunk of the token's int16 x, once for every task
        const bool hoist = FMT == kFmtQ2K && MAXT == 1 && nch == 1;
        typename FO::Frag fx;
        typename FO::Chunk pg, pu;  // the next item's words, in flight
        if (ok && q < q_et) {  // the first task's rows, requested before the L2 requests below
            if (hoist) FO::load_frag(xqf + (size_t)c0 * kFragWords, fx);
            const uint8_t* gr = task_row(task_pos(q));
            FO::load(gr + (c0 >> 2) * FO::kBlock, c0 & 3, pg);
            FO::load(gr + up_off + (c0 >> 2) * FO::kBlock, c0 & 3, pu);
        }
        // every routed gate/up row and every routed down row this CTA will read, requested into L2
        // at once, one 128-byte line per consumer thread at a time (gate/up lines first, in task order)
        {
            const int lines_gu = (L.rpw * L.rowH + 127) / 128;  // per task and matrix (its rows are contiguous)
            const int n_gu = q_et * 2 * lines_gu;
            const int64_t down_off = 2ll * P.F * L.rowH;
            const int lines_d = (P.RD * L.rowF + 127) / 128 + 1;  // + 1: the rows need not start on a line
            const int n_d = own_dg * na * lines_d;
            const int f_et = first_owned(L.n_ind, L.G, L.cta), f_dg = first_owned(lo_dg, L.G, L.cta);
            const FDiv d_l2 = fdiv_of(2 * lines_gu), d_ept = fdiv_of(L.ept), d_tpe = fdiv_of(L.tpe),
                       d_ld = fdiv_of(lines_d), d_na = fdiv_of(na > 0 ? na : 1);
#pragma unroll 1
            for (int i = tid; ok && i < n_gu + n_d; i += kCT) {
                const uint8_t* p;
                if (i < n_gu) {
                    int l, rt, tt;
                    const int q = fdiv(i, d_l2, l);
                    const int m = fdiv(q, d_ept, rt);
                    const int idx = f_et + m * L.G - L.n_ind;
                    const int a = fdiv(idx, d_tpe, tt);
                    const bool up = l >= lines_gu;
                    p = P.experts + (int64_t)C.act_e[a] * P.stride + (int64_t)(tt * P.R + rt * L.rpw) * L.rowH +
                        (up ? (int64_t)P.F * L.rowH : 0) + (int64_t)(up ? l - lines_gu : l) * 128;
                } else {
                    const int j = i - n_gu;
                    int l, a;
                    const int q = fdiv(j, d_ld, l);
                    const int m = fdiv(q, d_na, a);
                    const int r0 = (f_dg + m * L.G - lo_dg) * P.RD;
                    const uint8_t* row0 = P.experts + (int64_t)C.act_e[a] * P.stride + down_off + (int64_t)r0 * L.rowF;
                    const uint8_t* lim = row0 + (int64_t)P.RD * L.rowF;
                    p = row0 + (int64_t)l * 128;
                    if (p >= lim) p = lim - 1;  // the last line lands on the range's last byte
                }
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
            }
        }
        if (ok && q < q_et) {
            TaskPos cur = task_pos(q), nxt = cur;
            task_next(nxt);
            int n_done = 0;
#pragma unroll 1
            for (; q < q_et; q += kCW) {
                const int a = cur.a, tt = cur.tt;
                const int r = cur.rt * L.rpw + rl;
                const uint8_t* grow = task_row(cur);
                // one token: active expert a holds sorted entry a and no other
                const int j0 = MAXT == 1 ? a : C.act_begin[a], ne = MAXT == 1 ? 1 : C.act_begin[a + 1] - j0;
                float gacc[MAXT], uacc[MAXT];
#pragma unroll
                for (int e = 0; e < MAXT; e++) gacc[e] = uacc[e] = 0.0f;
#pragma unroll 1
                for (int i = 0; i < nch; i++) {
                    const int c = c0 + i * cstep;
                    const typename FO::Chunk gc = pg, uc = pu;
                    // request the next item: this task's next chunk, or the next task's first
                    if (i + 1 < nch) {
                        const uint8_t* gr = grow + ((c + cstep) >> 2) * FO::kBlock;
                        FO::load(gr, (c + cstep) & 3, pg);
                        FO::load(gr + up_off, (c + cstep) & 3, pu);
                    } else if (q + kCW < q_et) {
                        const uint8_t* gr = task_row(nxt) + (c0 >> 2) * FO::kBlock;
                        FO::load(gr, c0 & 3, pg);
                        FO::load(gr + up_off, c0 & 3, pu);
                    }
                    if (hoist) {
                        if (ne > 0) {
                            gacc[0] += FO::dot(gc, c & 3, fx);
                            uacc[0] += FO::dot(uc, c & 3, fx);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < MAXT; e++) {
                            if (e < ne) {
                                const int t = MAXT == 1 ? 0 : C.es_tok[j0 + e];
                                float dg, du;
                                FO::dot2(gc, uc, c & 3, xqf + ((size_t)t * (H / 64) + c) * kFragWords, dg, du);
                                gacc[e] += dg;
                                uacc[e] += du;
                            }
                        }
                    }
                }
#pragma unroll
                for (int e = 0; e < MAXT; e++) {
                    if (e < ne) {
                        float gv = gacc[e], uv = uacc[e];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            if (o < L.cpr) {
                                gv += __shfl_xor_sync(gm, gv, o);
                                uv += __shfl_xor_sync(gm, uv, o);
                            }
                        }
                        if (c0 == 0) {
                            const float sx = C.xscale[MAXT == 1 ? 0 : C.es_tok[j0 + e]] * (1.0f / 32767.0f);
                            P.xh[(size_t)(j0 + e) * F + tt * P.R + r] = silu(gv * sx) * (uv * sx);
                        }
                    }
                }
                n_done++;
                cur = nxt;
                task_next(nxt);
            }
            // the warp whose tasks complete the CTA's count publishes all of the CTA's h tiles.  Once
            // per warp, after its last task: a fence waits for the warp's loads in flight too, and
            // one per task would stall every next task's rows
            __syncwarp();  // orders the lanes' h stores before lane 0's fences below
            if (lane == 0) {
                __threadfence_block();
                if (atomicSub(&C.et_left, n_done) == n_done) {
                    __threadfence_block();
                    publish(C, ctr_h, kPubH);
                }
            }
        }
        // ---------------------------------------------------------- down rows: setup
        // This warp's down items (task, pass) form one stream, loaded two items ahead (four at one
        // token, where passes go in pairs).  The first ones depend only on the routing: they are
        // requested before the staging tasks and the waits for the staged h.
        const int al = L.cpf >= 32 ? 0 : lane / L.cpf;  // epp experts per pass, cpf lanes per expert row
        const int dc0 = L.cpf >= 32 ? lane : lane % L.cpf;
        const unsigned dgm = L.cpf >= 32 ? 0xffffffffu : (((1u << L.cpf) - 1u) << (lane & ~(L.cpf - 1)));
        const int du = dc0 & 3;
        const int np = (na + L.epp - 1) / L.epp;
        const int f_dg = first_owned(lo_dg, L.G, L.cta);
        float* pb = pbuf + warp * kMaxEnt;
        const int64_t dbase = 2ll * P.F * L.rowH + (dc0 >> 2) * FO::kBlock;  // this lane's bytes of a down row
        const int rd_sh = __ffs(P.RD) - 1;  // RD is a power of two
        auto drow = [&](int qq) -> int {  // output row of down task qq
            const int dq = qq - q_et - n_stage_tasks;
            return (f_dg + (dq >> rd_sh) * L.G - lo_dg) * P.RD + (dq & (P.RD - 1));
        };
        int iq = q, ip = 0;  // next item to request
        while (iq < q_et + n_stage_tasks) iq += kCW;
        int irow = iq < q_all ? drow(iq) : 0;  // its task's output row
        auto load_item = [&](typename FO::Chunk& dst) {
            if (iq >= q_all) return;
            const int row = irow;
            if (ip == 0 && S > 0 && lane * 128 < S * 2) {  // the task's shared down row, into L1
                const uint16_t* srow = P.sd + (size_t)row * S;
                for (int l = lane; l * 128 < S * 2; l += 32) asm volatile("prefetch.global.L1 [%0];" ::"l"(srow + l * 64));
            }
            const int a = ip * L.epp + al;
            if (a < na) FO::load(C.act_w[a] + dbase + (int64_t)row * L.rowF, du, dst);
            if (++ip == np) {
                ip = 0;
                iq += kCW;
                if (iq < q_all) irow = drow(iq);
            }
        };
        typename FO::Chunk b0{}, b1{}, b2{}, b3{};
        if (ok) {
            load_item(b0);
            load_item(b1);
            if (MAXT == 1) {  // one token: the stream runs two pass pairs ahead
                load_item(b2);
                load_item(b3);
            }
        }
        // ---------------------------------------------------------- staging of hs / of one entry's int16 h
#pragma unroll 1
        for (; ok && q < q_et + n_stage_tasks; q += kCW) {
            const int sidx = q - q_et;
            // the int16 h cache aliases x, w_sg and the int16 x fragments: wait until group B is
            // done with x and w_sg; the fragments' last reader, this CTA's last routed gate/up
            // task, ends before the CTA publishes its h, so entries are staged only after the
            // h counter below
            if (!(ok = warp_wait_mbar(C, &C.xq_bar, 0))) break;
            if (!(ok = warp_wait_mbar(C, &C.shared_bar, 0))) break;
            if (S > 0 && sidx == 0) {
                int got = 1;
                if (lane == 0) got = wait_count(ctr_hs, C.target, &C.abort);
                got = __shfl_sync(0xffffffffu, got, 0);
                __syncwarp();
                if (!(ok = got != 0)) break;
#pragma unroll 4
                for (int i = lane * 4; i < T * S; i += 128)
                    *reinterpret_cast<float4*>(hsf + i) = ld_relaxed_f32x4(P.xhs + i);
                __syncwarp();
                if (lane == 0) mbar_arrive(&C.hs_bar);
            } else {
                const int ent = sidx - (S > 0 ? 1 : 0);  // sorted position
                // the first entry task to get here waits for the h counter; the others for its flag
                int got = 1;
                if (lane == 0 && atomicCAS(&C.h_poller, 0, 1) == 0) {
                    got = wait_count(ctr_h, C.target, &C.abort);
                    if (got) mbar_arrive(&C.h_bar);
                }
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!(ok = got != 0 && warp_wait_mbar(C, &C.h_bar, 0))) break;
                const float* hr = P.xh + (size_t)ent * F;
                uint32_t* row = hqf + (size_t)ent * (F / 64) * kFragWords;
                // lane: 8 consecutive values per 256; the max-abs scale, then int16 fragments
                auto put8 = [&](int p, const float (&hv)[8], float inv) {
                    uint32_t wq[4];
                    int sum = 0;
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const int a0 = __float2int_rn(hv[2 * q] * inv);
                        const int a1 = __float2int_rn(hv[2 * q + 1] * inv);
                        wq[q] = (uint32_t)(a0 & 0xffff) | ((uint32_t)a1 << 16);
                        sum += a0 + a1;
                    }
                    FO::put8(row, p, wq, sum, true);
                };
                auto load8f = [&](int p, float (&hv)[8]) {
                    const float4 a = ld_relaxed_f32x4(hr + p), b = ld_relaxed_f32x4(hr + p + 4);
                    hv[0] = a.x; hv[1] = a.y; hv[2] = a.z; hv[3] = a.w;
                    hv[4] = b.x; hv[5] = b.y; hv[6] = b.z; hv[7] = b.w;
                };
                auto absmax8 = [](const float (&hv)[8], float m) {
#pragma unroll
                    for (int i = 0; i < 8; i++) m = fmaxf(m, fabsf(hv[i]));
                    return m;
                };
                float m = 0.0f;
                if (MAXT > 1 && F <= 1024) {  // one pass over L2: the row stays in registers (measured: one
                                              // token is faster with two passes)
                    float hv[4][8];
#pragma unroll
                    for (int it = 0; it < 4; it++)
                        if (it * 256 < F) load8f(lane * 8 + it * 256, hv[it]);
#pragma unroll
                    for (int it = 0; it < 4; it++)
                        if (it * 256 < F) m = absmax8(hv[it], m);
                    m = warp_max(m);
                    const float inv = m > 0.0f ? 32767.0f / m : 0.0f;
#pragma unroll
                    for (int it = 0; it < 4; it++)
                        if (it * 256 < F) put8(lane * 8 + it * 256, hv[it], inv);
                } else {  // two passes
#pragma unroll 2
                    for (int p = lane * 8; p < F; p += 256) {
                        float hv[8];
                        load8f(p, hv);
                        m = absmax8(hv, m);
                    }
                    m = warp_max(m);
                    const float inv = m > 0.0f ? 32767.0f / m : 0.0f;
#pragma unroll 2
                    for (int p = lane * 8; p < F; p += 256) {
                        float hv[8];
                        load8f(p, hv);
                        put8(p, hv, inv);
                    }
                }
                if (lane == 0) C.hscale[ent] = m * (1.0f / 32767.0f);
                __syncwarp();
                if (lane == 0) mbar_arrive(&C.staged_bar);
            }
        }
        // ---------------------------------------------------------- down rows
        if (ok && q < q_all) {
            if (S > 0) ok = warp_wait_mbar(C, &C.hs_bar, 0);
            if (ok) ok = warp_wait_mbar(C, &C.staged_bar, 0);
        }
#pragma unroll 1
        for (; ok && q < q_all; q += kCW) {
            const int row = drow(q);
            if (MAXT == 1) {
                // one token: one entry per active expert; two passes at a time, their two dot
                // chains independent (the same sums, the same order)
#pragma unroll 1
                for (int pa = 0; pa < np; pa += 2) {
                    const bool two = pa + 1 < np;  // the stream holds passes pa, pa + 1 in b0, b1
                    typename FO::Chunk n0{}, n1{};
                    load_item(n0);
                    if (two) load_item(n1);
                    const int a0 = pa * L.epp + al, a1 = a0 + L.epp;
                    const bool h0 = a0 < na, h1 = two && a1 < na;
                    const int j0 = h0 ? a0 : 0, j1 = h1 ? a1 : 0;  // one entry per active expert
                    float v0 = 0.0f, v1 = 0.0f;
                    if (h0) {
                        typename FO::Frag f0;
                        FO::load_frag(hqf + ((size_t)j0 * (F / 64) + dc0) * kFragWords, f0);
                        v0 = FO::dot(b0, du, f0);
                    }
                    if (h1) {
                        typename FO::Frag f1;
                        FO::load_frag(hqf + ((size_t)j1 * (F / 64) + dc0) * kFragWords, f1);
                        v1 = FO::dot(b1, du, f1);
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        if (o < L.cpf) {
                            v0 += __shfl_xor_sync(dgm, v0, o);
                            v1 += __shfl_xor_sync(dgm, v1, o);
                        }
                    }
                    if (dc0 == 0) {
                        if (h0) pb[j0] = v0 * C.hscale[j0];
                        if (h1) pb[j1] = v1 * C.hscale[j1];
                    }
                    if (two) {
                        b0 = b2;
                        b1 = b3;
                        b2 = n0;
                        b3 = n1;
                    } else {  // b1 already holds the next task's first item
                        b0 = b1;
                        b1 = b2;
                        b2 = b3;
                        b3 = n0;
                    }
                }
            } else {
#pragma unroll 1
            for (int pa = 0; pa < np; pa++) {
                load_item(b2);
                const int a = pa * L.epp + al;
                if (a < na) {
                    // the expert's entries two at a time: two independent dot chains against one
                    // chunk (the same sums, the same order)
                    const int je = C.act_begin[a + 1];
#pragma unroll 1
                    for (int j = C.act_begin[a]; j < je; j += 2) {
                        const bool two = j + 1 < je;  // uniform over the lanes of this expert's row
                        float v0, v1 = 0.0f;
                        {
                            typename FO::Frag f;
                            FO::load_frag(hqf + ((size_t)j * (F / 64) + dc0) * kFragWords, f);
                            v0 = FO::dot(b0, du, f);
                        }
                        if (two) {
                            typename FO::Frag f;
                            FO::load_frag(hqf + ((size_t)(j + 1) * (F / 64) + dc0) * kFragWords, f);
                            v1 = FO::dot(b0, du, f);
                        }
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            if (o < L.cpf) {
                                v0 += __shfl_xor_sync(dgm, v0, o);
                                v1 += __shfl_xor_sync(dgm, v1, o);
                            }
                        }
                        if (dc0 == 0) {
                            pb[j] = v0 * C.hscale[j];
                            if (two) pb[j + 1] = v1 * C.hscale[j + 1];
                        }
                    }
                }
                b0 = b1;
                b1 = b2;
            }
            }
            // shared expert down row
            float sacc[MAXT];
            if (S > 0)
                warp_dense_row<MAXT>(reinterpret_cast<const uint8_t*>(P.sd + (size_t)row * S), false, S,
                                     reinterpret_cast<const uint8_t*>(hsf), true, T, sacc);
            __syncwarp();
#pragma unroll
            for (int t = 0; t < MAXT; t++) {
                if (t < T && lane == t) {
                    float acc = 0.0f;
                    if (MAXT == 1) {  // one token: its entries are sorted positions 0 .. k-1
#pragma unroll 8
                        for (int j = 0; j < k; j++) acc = fmaf(C.ps[j], pb[j], acc);
                    } else {
#pragma unroll 1
                        for (int mm = 0; mm < k; mm++) {
                            const int j = C.tok_sorted[t * k + mm];
                            acc = fmaf(C.ps[j], pb[j], acc);
                        }
                    }
                    if (S > 0) acc = fmaf(C.gate_s[t], sacc[t], acc);
                    P.out[(size_t)t * H + row] = acc;
                }
            }
        }
        if (!ok) fail(C, status);
    }

    __syncthreads();
    if (tid == 0) {
        // never leave a copy in flight into shared memory that is about to be released
        const int issued = vload(&C.issued);
#pragma unroll 1
        for (int s = max(0, issued - ns); s < issued; s++)
            if (!mbar_wait(&C.full[s % ns], (s / ns) & 1)) set_status(status, QS_ERR_TIMEOUT);
        if (!mbar_wait(&C.xbar, 0)) set_status(status, QS_ERR_TIMEOUT);
        if (vload(&C.abort)) set_status(status, QS_ERR_TIMEOUT);
        // keep every counter at exactly gridDim per call, whatever happened
        const int pub = vload(&C.published);
        if (!(pub & kPubLogits)) red_relaxed_add_u64(ctr_lg, 1);
        if (!(pub & kPubHs)) red_relaxed_add_u64(ctr_hs, 1);
        if (!(pub & kPubH)) red_relaxed_add_u64(ctr_h, 1);
        red_relaxed_add_u64(ctr_exit, 1);
    }
}

// ------------------------------------------------------------------ host side

static bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
static size_t up16(size_t v) { return (v + 15) / 16 * 16; }

struct FusedPlanHost {
    int RR, RS, R, RD, nstages, sg_direct;
    int off_xq, off_sig, off_hsf, off_hq, off_pbuf, off_stages;
    size_t smem;
};

static bool plan_fused(const qs_moe_shape& s, int T, int n_sm, size_t smem_max, FusedPlanHost& fp) {
    const int H = s.hidden, E = s.n_experts, k = s.top_k, F = s.expert_ffn, S = s.shared_ffn;
    const int nbH = H / 256, nbF = F / 256;
    const int xsz = s.x_dtype == QS_BF16 ? 2 : 4;
    if (T < 1 || T > kMaxT || T * k > kMaxEnt || T > 32) return false;
    if (T * ((E + 31) / 32) * std::min(k, 32) > kMaxCand) return false;
    if (!pow2(nbH) || nbH > 32 || !pow2(nbF) || 4 * nbF > 32) return false;
    if (S > 0 && (!pow2(S / 256) || S / 256 > 32)) return false;
    if (H * 4 > kStageBytes) return false;            // a router row must fit a stage
    if (S > 0 && 4 * H > kStageBytes) return false;    // a shared gate+up row pair must fit
    fp.RR = std::min(E, kStageBytes / (H * 4));
    while (E % fp.RR) fp.RR--;
    fp.RS = 0;
    if (S > 0) {
        fp.RS = kStageBytes / (4 * H);
        while (S % fp.RS) fp.RS--;
    }
    fp.R = 128 / nbH;
    const int rd_align = 4 / std::min(nbF, 4);
    int RD = kMaxRD;
    // down groups of RD output rows: at least four per CTA (their rows are loaded from global
    // memory by the warps that use them, not staged)
    while (RD > rd_align && H / RD < 4 * n_sm) RD /= 2;
    while (RD > H) RD /= 2;
    if (RD < rd_align || H % RD) return false;
    fp.RD = RD;
    // region 0: x as given, w_sg and the int16 x fragments -- later the int16 h cache (x and
    // w_sg are dead once group B has finished its shared gate/up rows; the x fragments once this
    // CTA's last routed gate/up task has ended, which is before the CTA publishes its h)
    size_t o = up16((size_t)T * H * xsz);
    fp.off_sig = (int)o;
    o += up16((size_t)H * 2);
    fp.off_xq = (int)o;
    o += up16((size_t)T * (H / 64) * kFragWords * 4);
    fp.off_hq = 0;
    o = std::max(o, up16((size_t)T * k * (F / 64) * kFragWords * 4));
    fp.off_hsf = (int)o;
    o += up16((size_t)T * S * 4);
    fp.off_pbuf = (int)o;
    o += (size_t)kCW * kMaxEnt * 4;
    o = (o + 127) / 128 * 128;
    fp.off_stages = (int)o;
    const size_t fixed = (sizeof(FusedCtl) + 127) / 128 * 128 + o;
    if (fixed + (size_t)kStageBytes > smem_max) return false;  // one stage at least (router and shared rows)
    fp.nstages = (int)std::min<size_t>(kMaxStages, (smem_max - fixed) / kStageBytes);
    fp.smem = fixed + (size_t)fp.nstages * kStageBytes;
    // the shared gate/up rows go through the ring when it is deep enough for several tokens;
    // for one token, or a ring of one or two stages, group B reads them from global memory
    // (measured: 35B-A3B layer 0.45 us faster at one token, 2.4-3.6 us slower at four and eight
    // through global memory; H=4096 layer with one stage at four tokens 66 us faster)
    fp.sg_direct = (T == 1 || fp.nstages < 3) ? 1 : 0;
    return true;
}

// Per-device facts the launcher needs on every call, read once per device.
struct DeviceFacts {
    int n_sm = 0, smem_max = 0;
    size_t smem_set[8] = {};  // dynamic smem limit set per kernel instantiation
};
constexpr int kMaxDevices = 64;
static DeviceFacts g_dev[kMaxDevices];

static cudaError_t device_facts(DeviceFacts** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    DeviceFacts& f = g_dev[dev];
    if (f.n_sm == 0) {
        int n = 0, m = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        f.smem_max = m;
        f.n_sm = n;
    }
    *out = &f;
    return cudaSuccess;
}

template <int MAXT, int FMT, int SLOT>
static cudaError_t launch_fused_t(const FusedParams& p, size_t smem, DeviceFacts& f, cudaStream_t st) {
    const void* fn = (const void*)fused_decode_kernel<MAXT, FMT>;
    if (f.smem_set[SLOT] < smem) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        f.smem_set[SLOT] = smem;
    }
    FusedParams pp = p;
    // Not a cooperative launch: that would serialise this call behind the previous one.  The
    // grid is one CTA per SM and nothing else in the stream runs beside it, so every CTA is
    // resident; if other work held SMs longer than the wait bound, the call ends in a time-out.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(f.n_sm);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_decode_kernel<MAXT, FMT>, pp);
}

bool fused_decode_supported(const qs_moe_shape& s, int T, cudaError_t* err) {
    DeviceFacts* f = nullptr;
    *err = device_facts(&f);
    if (*err != cudaSuccess) return false;
    FusedPlanHost fp;
    return plan_fused(s, T, f->n_sm, (size_t)f->smem_max, fp);
}

// Returns cudaErrorNotSupported when the shape is outside the fused kernel's plan.
cudaError_t launch_fused_decode(const qs_moe_shape& s, const void* x, const float* Wr, const float* bias,
                                const uint8_t* experts, int64_t stride, const uint16_t* sg, const uint16_t* su,
                                const uint16_t* sd, const uint16_t* ssig, int T, float* out, void* ws,
                                const WsLayout& W, cudaStream_t st, bool x_host_mapped, int fmt) {
    DeviceFacts* f = nullptr;
    cudaError_t e = device_facts(&f);
    if (e != cudaSuccess) return e;
    FusedPlanHost fp;
    if (!plan_fused(s, T, f->n_sm, (size_t)f->smem_max, fp)) return cudaErrorNotSupported;
    FusedParams p;
    p.x = x;
    p.Wr = Wr;
    p.bias = bias;
    p.experts = experts;
    p.stride = stride;
    p.sg = sg;
    p.su = su;
    p.sd = sd;
    p.ssig = ssig;
    p.out = out;
    uint8_t* base = static_cast<uint8_t*>(ws);
    p.xlog = reinterpret_cast<float*>(base + W.xlog);
    p.xhs = reinterpret_cast<float*>(base + W.xhs);
    p.xh = reinterpret_cast<float*>(base + W.xh);
    p.rec_ids = reinterpret_cast<int32_t*>(base + W.ids);
    p.rec_p = reinterpret_cast<float*>(base + W.pw);
    p.hdr = reinterpret_cast<WsHeader*>(base + W.header);
    p.H = s.hidden;
    p.E = s.n_experts;
    p.k = s.top_k;
    p.F = s.expert_ffn;
    p.S = (sg != nullptr) ? s.shared_ffn : 0;
    p.T = T;
    p.x_dtype = s.x_dtype;
    p.RR = fp.RR;
    p.RS = fp.RS;
    p.R = fp.R;
    p.RD = fp.RD;
    p.nstages = fp.nstages;
    p.sg_direct = fp.sg_direct;
    p.x_sys = x_host_mapped ? 1 : 0;
    p.off_xq = fp.off_xq;
    p.off_sig = fp.off_sig;
    p.off_hsf = fp.off_hsf;
    p.off_hq = fp.off_hq;
    p.off_pbuf = fp.off_pbuf;
    p.off_stages = fp.off_stages;
    if (fmt == kFmtQ4K) {
        if (T == 1 && s.top_k <= 32) return launch_fused_t<1, kFmtQ4K, 4>(p, fp.smem, *f, st);
        if (T <= 4) return launch_fused_t<4, kFmtQ4K, 5>(p, fp.smem, *f, st);
        if (T <= 8) return launch_fused_t<8, kFmtQ4K, 6>(p, fp.smem, *f, st);
        return launch_fused_t<16, kFmtQ4K, 7>(p, fp.smem, *f, st);
    }
    if (T == 1 && s.top_k <= 32) return launch_fused_t<1, kFmtQ2K, 0>(p, fp.smem, *f, st);
    if (T <= 4) return launch_fused_t<4, kFmtQ2K, 1>(p, fp.smem, *f, st);
    if (T <= 8) return launch_fused_t<8, kFmtQ2K, 2>(p, fp.smem, *f, st);
    return launch_fused_t<16, kFmtQ2K, 3>(p, fp.smem, *f, st);
}

}  // namespace qs

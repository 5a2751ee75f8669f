// qs_cluster.cu -- the decode-sized MoE-FFN layer as one kernel of thread-block clusters (sm_103a).
//
// The layer (QuarkStar (q36) README, "Model Weights": routed experts 2-bit, shared expert and
// router in higher precision; Quasar (q27) README, "Design decisions": dequantisation fused into
// the GEMV) for a few tokens per call.  The grid is NCL clusters of kCS = 8 CTAs, one CTA per SM,
// every CTA resident at once.  A cluster owns whole routed experts ("units"): its 8 CTAs each
// compute F/8 of the expert's gate/up rows, hand their slice of h = silu(Wg x)*(Wu x) to every
// CTA of the cluster through distributed shared memory, and then each CTA forms the expert's
// down product over its H/8 output rows.  So h never leaves the cluster; the only grid-wide
// exchanges are the router logits (before top-k) and the shared expert's hs.
//
// Per CTA (g = cluster * 8 + rank), in order:
//   static rows, requested at kernel start (before the previous kernel in the stream has
//   finished: weights are never written by a running kernel):  its share of the router rows,
//   of the shared expert's gate/up rows and of the shared expert's down rows of slice `rank`
//   (output rows [rank*H/8, (rank+1)*H/8) are slice `rank`);
//   x (after griddepcontrol.wait) -> per-token int16 x, its max-abs scale, the sigmoid gate;
//   router rows -> logits (global), publish;
//   wait for every CTA's logits -> top-k + softmax for every token (every CTA, identically),
//   active experts ascending; unit u (the u-th active expert) belongs to cluster u % NCL;
//   the routed rows of the cluster's units are requested now;
//   shared gate/up rows (already in shared memory) -> hs (global), publish;
//   per unit: gate/up rows (rows [rank*F/8, ...)) -> h slice -> every peer's shared memory;
//   wait for the 8 slices -> per-entry max-abs int16 h -> down rows of slice `rank` ->
//   pd[entry][row] (global);
//   wait for every CTA's hs -> shared down rows (requested after the routed rows) ->
//   sdp[t][row] (global);
//   ticket of slice `rank` (+1 per CTA per call): the CTA completing it adds, for every token
//   and row of the slice, sum over the token's slots of p * pd, then gate * sdp -> out.
//
// Weight bytes move by bulk asynchronous copies (TMA engine, 1-D) into a ring of stages; one
// producer warp issues them, 16 consumer warps walk the same sequence of stages.  Grid-wide
// counters are 64-bit and never reset: every call adds exactly gridDim to the logits, hs and
// exit counters and NCL to each slice ticket, whatever happens, so call n's targets follow
// from the exit count read after griddepcontrol.wait.  Every wait is bounded by the global
// timer; one that runs out records QS_ERR_TIMEOUT in the status word and the CTA winds down,
// still adding what it owes to every counter, letting its copies land and meeting its cluster
// at the final cluster barrier.
#include "qs_common.cuh"
#include "qs_internal.h"
#include "qs_q2k.cuh"
#include "qs_warp.cuh"

#include <algorithm>
#include <mutex>

namespace qs {
namespace {

constexpr int kCS = kClusterCtas;    // CTAs per cluster
constexpr int kCW = 15;              // consumer warps (with the producer, 16 warps: 128 registers a thread)
constexpr int kCT = kCW * 32;
constexpr int kThreads = kCT + 32;   // + the producer warp
constexpr int kSB = 21504;           // stage bytes (256 Q2_K blocks)
constexpr int kMaxNS = 12;
constexpr int kMaxT = kClusterMaxT;
constexpr int kMaxEnt = 64;          // T * k
constexpr int kBarCons = 1;          // named barrier of the consumer warps
constexpr int kMaxItems = 48;        // dense rows (or row segments) of one stage
constexpr bool kHoistX = true;       // one token: keep the lane's x fragment in registers (gate/up)
constexpr bool kHoistH = true;       // ... and its h fragment (down)
static_assert(kMaxT == 8, "dense-stage epilogues map a thread to (row, token) as (tid >> 3, tid & 7)");

// counters, one per 32-byte sector of the counter region
enum { kCxLogits = 0, kCxHs = 1, kCxExit = 2, kCxTicket = 3 };
enum { kPubLogits = 1, kPubHs = 2, kPubTicket = 4 };

struct CParams {
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
    float* logits;     // [T x E]
    float* hs;         // [T x S]
    float* pd;         // [T*k x H]  routed down products per entry (unweighted)
    float* sdp;        // [T x H]    shared down products (ungated)
    int32_t* rec_ids;  // [T*k]      the routing of the call (written by CTA 0)
    float* rec_p;      // [T*k]
    uint8_t* cx;       // counters
    uint32_t* status;
    int H, E, k, F, S, T, x_dtype;
    int x_sys;         // x is host memory reached through its mapped address: the consumers load it
    int NCL;
    int ns;
    int rr, ps, dsr, gp, dr;  // per stage: router rows, shared gate/up pairs, shared down rows, routed pairs, routed down rows
    int off_x, off_sig, off_xq, off_hbuf, off_hq, off_uraw, off_stages;
    int hbuf_bytes;
    // geometry, computed on the host
    int lgH;          // log2 H
    int rowH, rowF;   // Q2_K row bytes along H (gate/up rows) and along F (down rows)
    int cpr, cpf;     // 64-weight chunks per gate/up row and per down row
    int gsz, rpw;     // gate/up: lanes per row (<= 32) and rows per warp pass
    int drpw;         // down: rows per warp pass (cpf lanes per row)
    int PR, HS;       // gate/up rows and down rows of one unit per CTA
    int lgper;        // log2 of the float4s in a CTA's slice of one entry's h (PR / 4)
};

struct alignas(16) CCtl {
    uint64_t full[kMaxNS];
    uint64_t empty[kMaxNS];
    uint64_t xbar;        // x and w_sg landed
    uint64_t routed_bar;  // routing published (the producer waits on it)
    uint64_t hx[2];       // the cluster's h slices of a unit landed (kCS arrivals)
    uint64_t target_g;    // this call's target of the logits / hs counters
    uint64_t target_t;    // ... and of the slice tickets
    int abort, issued, n_act, last;
    int pub, n_ent, pad0, pad1;
    int ids[kMaxEnt];
    float p[kMaxEnt];
    int ent_sorted[kMaxEnt];   // entries t*k+slot ordered by (expert, entry)
    int es_tok[kMaxEnt];       // token of ent_sorted[i]
    int act_e[kMaxEnt];        // active experts, ascending
    int act_begin[kMaxEnt + 1];
    float xscale[kMaxT];
    float gate_s[kMaxT];
    float hscale[kMaxT];       // current unit's per-entry h scales
    float part[2][kMaxItems][kMaxT];  // per-warp partial dot products of a stage's dense rows
};

__device__ __forceinline__ uint64_t* cx_ctr(const CParams& P, int i) {
    return reinterpret_cast<uint64_t*>(P.cx + 32 * i);
}

__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync %0, %1;" ::"n"(kBarCons), "n"(kCT) : "memory"); }

// Position in the ring of stages: slot and the parity of its current fill.
struct Ring {
    int slot;
    uint32_t ph;
    __device__ __forceinline__ void next(int ns) {
        if (++slot == ns) {
            slot = 0;
            ph ^= 1u;
        }
    }
};

// ------------------------------------------------------------------ cluster primitives

__device__ __forceinline__ uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// The address of this CTA's shared-memory word `local` in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cl_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void fence_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }
// Arrive (release at cluster scope) on the mbarrier at cluster address `addr`.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
// Phase test with acquire at cluster scope (sees the peers' stores released by their arrivals).
__device__ __forceinline__ bool mbar_test_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// As above; the thread may be suspended up to hint_ns while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

__device__ __forceinline__ uint64_t atom_add_acq_rel_u64(uint64_t* p, uint64_t v) {
    uint64_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}

// ------------------------------------------------------------------ bounded waits

__device__ __forceinline__ void fail(CCtl& C, uint32_t* status) {
    set_status(status, QS_ERR_TIMEOUT);
    vstore(&C.abort, 1);
}

// Whole warp waits for an mbarrier phase: try_wait blocks in hardware for a while and returns
// as soon as the phase completes; the abort flag and the time limit are looked at every 16
// polls.  False on abort or time-out (then the CTA is marked aborting).  Not inlined: one copy
// of the code serves every wait of the kernel.
__device__ __noinline__ bool warp_wait(CCtl& C, uint64_t* bar, uint32_t parity, uint32_t* status, int cluster_scope) {
    bool ok = true;
    if (!(cluster_scope ? mbar_test_cluster(bar, parity) : mbar_try_wait(bar, parity))) {
        const uint64_t t0 = global_timer_ns();
#pragma unroll 1
        for (int it = 1;; it++) {
            if (cluster_scope ? mbar_test_cluster(bar, parity) : mbar_try_wait(bar, parity)) break;
            if ((it & 15) == 0 && (vload(&C.abort) || global_timer_ns() - t0 > kWaitNs)) {
                ok = false;
                break;
            }
        }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0) fail(C, status);
    return ok && !vload(&C.abort);
}

// One thread: wait with acquire loads until counter *c reaches target.
__device__ __forceinline__ bool wait_count(const uint64_t* c, uint64_t target, const int* abort) {
    if (ld_acquire_u64(c) >= target) return true;
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_u64(c) < target) {
        if (*reinterpret_cast<const volatile int*>(abort) || global_timer_ns() - t0 > kWaitNs) return false;
    }
    return true;
}

// ------------------------------------------------------------------ dense rows of a stage

// Dot products of the n rows at `w` (K elements each, fp32 if w_f32 else bf16) with the T
// activation rows at `act` ([T x K], fp32 if a_f32 else bf16), spread over the consumer warps:
// with n < kCW rows each row is cut into nseg = kCW / n segments of whole 256-element blocks,
// one per warp.  Item it = row * nseg + segment; its warp sum per token goes to part[it][t].
// Returns nseg.  The caller adds a row's segments in order (row_dot) after a consumer barrier.
template <int MAXT>
__device__ __forceinline__ int stage_dense(const uint8_t* w, bool w_f32, int K, int n, const uint8_t* act, bool a_f32,
                                           int T, float (*part)[kMaxT]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int lg = 0;  // nseg = 2^lg, the largest with n * nseg <= kCW
    while ((n << (lg + 1)) <= kCW) lg++;
    const int nseg = 1 << lg;
    const int nb = K / 256;
    const int wsz = w_f32 ? 4 : 2, asz = a_f32 ? 4 : 2;
#pragma unroll 1
    for (int it = warp; it < n * nseg; it += kCW) {
        const int r = it >> lg, sg = it & (nseg - 1);
        const int i1 = ((nb * (sg + 1)) >> lg) * 256;
        const uint8_t* row = w + (size_t)r * K * wsz;
        float acc[MAXT];
#pragma unroll
        for (int t = 0; t < MAXT; t++) acc[t] = 0.0f;
#pragma unroll 2
        for (int i = ((nb * sg) >> lg) * 256 + lane * 8; i < i1; i += 256) {
            float wv[8];
            load8(row + (size_t)i * wsz, w_f32, wv);
#pragma unroll
            for (int t = 0; t < MAXT; t++) {
                if (t < T) {
                    float av[8];
                    load8(act + ((size_t)t * K + i) * asz, a_f32, av);
                    float sum = acc[t];
#pragma unroll
                    for (int q = 0; q < 8; q++) sum = fmaf(wv[q], av[q], sum);
                    acc[t] = sum;
                }
            }
        }
#pragma unroll
        for (int t = 0; t < MAXT; t++) {
            if (t < T) {
                const float v = warp_sum(acc[t]);
                if (lane == 0) part[it][t] = v;
            }
        }
    }
    return nseg;
}

__device__ __forceinline__ float row_dot(const float (*part)[kMaxT], int r, int t, int nseg) {
    float v = 0.0f;
#pragma unroll 1
    for (int sg = 0; sg < nseg; sg++) v += part[r * nseg + sg][t];
    return v;
}

// ------------------------------------------------------------------ job sequence

enum JobKind { kJobRouter = 0, kJobSharedGU = 1, kJobSharedDown = 2, kJobGU = 3, kJobDown = 4 };

struct Job {
    int kind, e, r0, n;  // expert (routed jobs), first row, rows (pairs)
};

// This CTA's static row ranges and stage counts.
struct Statics {
    int r0, r1, nr;   // router rows
    int s0, s1, nsg;  // shared gate/up row pairs
    int d0, d1, nsd;  // shared down rows (of slice `rank`), requested after the routed rows
    int n;            // stages requested before the routing is known (router, shared gate/up)
    int ngu, ndn;     // stages of one routed unit: gate/up, down
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ Statics make_statics(const CParams& P, int g, int c, int rank) {
    Statics s;
    const int G = P.NCL * kCS;
    s.r0 = (int)((int64_t)P.E * g / G);
    s.r1 = (int)((int64_t)P.E * (g + 1) / G);
    s.nr = cdiv(s.r1 - s.r0, P.rr);
    s.s0 = P.S > 0 ? (int)((int64_t)P.S * g / G) : 0;
    s.s1 = P.S > 0 ? (int)((int64_t)P.S * (g + 1) / G) : 0;
    s.nsg = P.S > 0 ? cdiv(s.s1 - s.s0, P.ps) : 0;
    const int HS = P.HS;
    s.d0 = P.S > 0 ? rank * HS + HS * c / P.NCL : 0;
    s.d1 = P.S > 0 ? rank * HS + HS * (c + 1) / P.NCL : 0;
    s.nsd = P.S > 0 ? cdiv(s.d1 - s.d0, P.dsr) : 0;
    s.n = s.nr + s.nsg;
    s.ngu = cdiv(P.PR, P.gp);
    s.ndn = cdiv(HS, P.dr);
    return s;
}

__device__ __forceinline__ Job static_job(const CParams& P, const Statics& s, int i) {
    Job j;
    j.e = -1;
    if (i < s.nr) {
        j.kind = kJobRouter;
        j.r0 = s.r0 + i * P.rr;
        j.n = min(P.rr, s.r1 - j.r0);
    } else {
        j.kind = kJobSharedGU;
        j.r0 = s.s0 + (i - s.nr) * P.ps;
        j.n = min(P.ps, s.s1 - j.r0);
    }
    return j;
}

// Shared down job i (requested after every routed row of the cluster's units).
__device__ __forceinline__ Job shared_down_job(const CParams& P, const Statics& s, int i) {
    Job j;
    j.e = -1;
    j.kind = kJobSharedDown;
    j.r0 = s.d0 + i * P.dsr;
    j.n = min(P.dsr, s.d1 - j.r0);
    return j;
}

// Job i of one routed unit (expert e) for cluster rank `rank`.
__device__ __forceinline__ Job unit_job(const CParams& P, const Statics& s, int e, int rank, int i) {
    Job j;
    j.e = e;
    if (i < s.ngu) {
        j.kind = kJobGU;
        j.r0 = rank * P.PR + i * P.gp;
        j.n = min(P.gp, (rank + 1) * P.PR - j.r0);
    } else {
        j.kind = kJobDown;
        j.r0 = rank * P.HS + (i - s.ngu) * P.dr;
        j.n = min(P.dr, (rank + 1) * P.HS - j.r0);
    }
    return j;
}

// ------------------------------------------------------------------ producer

// One thread: wait for an mbarrier phase, watching the abort flag; false on abort or time-out.
__device__ __noinline__ bool thread_wait(CCtl& C, uint64_t* bar, uint32_t parity, uint32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    for (int it = 1; !mbar_try_wait(bar, parity); it++) {
        if ((it & 15) == 0) {
            if (vload(&C.abort)) return false;
            if (global_timer_ns() - t0 > kWaitNs) {
                fail(C, status);
                return false;
            }
        }
    }
    return true;
}

// The producer's position: the ring slot of the next copy, the parity of that slot's fill, and
// whether the ring has wrapped (from then on a slot is free once its previous fill is released).
struct PRing {
    int slot;
    uint32_t ph;
    bool wrapped;
    __device__ __forceinline__ void next(int ns) {
        if (++slot == ns) {
            slot = 0;
            ph ^= 1u;
            wrapped = true;
        }
    }
};

// lane 0: wait until the ring's next slot is free; false (abort) on time-out
__device__ __forceinline__ bool producer_free(CCtl& C, const CParams& P, const PRing& R) {
    if (!R.wrapped) return true;
    if (vload(&C.abort)) return false;
    return thread_wait(C, &C.empty[R.slot], R.ph ^ 1u, P.status);
}

__device__ __forceinline__ void producer_issue(CCtl& C, const CParams& P, uint8_t* stages, const PRing& R, const Job& j) {
    uint8_t* dst = stages + (size_t)R.slot * kSB;
    uint64_t* bar = &C.full[R.slot];
    const int rowH = P.rowH, rowF = P.rowF;
    fence_proxy_async_smem();
    switch (j.kind) {
        case kJobRouter: {
            const uint32_t b = (uint32_t)j.n * P.H * 4;
            mbar_arrive_expect_tx(bar, b);
            bulk_g2s(dst, P.Wr + (size_t)j.r0 * P.H, b, bar);
            break;
        }
        case kJobSharedGU: {
            const uint32_t b = (uint32_t)j.n * P.H * 2;
            mbar_arrive_expect_tx(bar, 2 * b);
            bulk_g2s(dst, P.sg + (size_t)j.r0 * P.H, b, bar);
            bulk_g2s(dst + b, P.su + (size_t)j.r0 * P.H, b, bar);
            break;
        }
        case kJobSharedDown: {
            const uint32_t b = (uint32_t)j.n * P.S * 2;
            mbar_arrive_expect_tx(bar, b);
            bulk_g2s(dst, P.sd + (size_t)j.r0 * P.S, b, bar);
            break;
        }
        case kJobGU: {
            const uint32_t b = (uint32_t)j.n * rowH;
            const uint8_t* ex = P.experts + (int64_t)j.e * P.stride;
            mbar_arrive_expect_tx(bar, 2 * b);
            bulk_g2s(dst, ex + (int64_t)j.r0 * rowH, b, bar);
            bulk_g2s(dst + b, ex + (int64_t)(P.F + j.r0) * rowH, b, bar);
            break;
        }
        default: {
            const uint32_t b = (uint32_t)j.n * rowF;
            const uint8_t* dn = P.experts + (int64_t)j.e * P.stride + 2ll * P.F * rowH;
            mbar_arrive_expect_tx(bar, b);
            bulk_g2s(dst, dn + (int64_t)j.r0 * rowF, b, bar);
            break;
        }
    }
}

__device__ void producer(CCtl& C, const CParams& P, uint8_t* data) {
    const int lane = threadIdx.x & 31;
    const int rank = (int)cl_rank(), c = (int)cl_id();
    const Statics s = make_statics(P, blockIdx.x, c, rank);
    uint8_t* stages = data + P.off_stages;
    int seq = 0;
    PRing R{0, 0u, false};
    if (lane == 0) {
        // routing-independent rows first, as many as there are free stages: weights, which no
        // running kernel writes, so they may be read before the previous kernel has finished
        const int first = min(s.n, P.ns);
        for (; seq < first; seq++, R.next(P.ns)) producer_issue(C, P, stages, R, static_job(P, s, seq));
        const uint32_t xb = (uint32_t)P.T * P.H * (P.x_dtype == QS_BF16 ? 2 : 4);
        const uint32_t sb = P.S > 0 ? (uint32_t)P.H * 2 : 0u;
        mbar_arrive_expect_tx(&C.xbar, (P.x_sys ? 0u : xb) + sb);
        if (sb) bulk_g2s(data + P.off_sig, P.ssig, sb, &C.xbar);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (!P.x_sys) bulk_g2s(data + P.off_x, P.x, xb, &C.xbar);
        for (; seq < s.n; seq++, R.next(P.ns)) {
            if (!producer_free(C, P, R)) goto done;
            producer_issue(C, P, stages, R, static_job(P, s, seq));
        }
        // the routed rows of this cluster's units, once the routing is known
        {
            if (vload(&C.abort) || !thread_wait(C, &C.routed_bar, 0, P.status)) goto done;
            const int n_act = vload(&C.n_act);
            for (int u = c; u < n_act; u += P.NCL) {
                const int e = C.act_e[u];
                for (int i = 0; i < s.ngu + s.ndn; i++, seq++, R.next(P.ns)) {
                    if (!producer_free(C, P, R)) goto done;
                    producer_issue(C, P, stages, R, unit_job(P, s, e, rank, i));
                }
            }
            for (int i = 0; i < s.nsd; i++, seq++, R.next(P.ns)) {
                if (!producer_free(C, P, R)) goto done;
                producer_issue(C, P, stages, R, shared_down_job(P, s, i));
            }
        }
    done:
        vstore(&C.issued, seq);
    }
    __syncwarp();
}

// ------------------------------------------------------------------ the kernel

template <int MAXT>
__global__ void __launch_bounds__(kThreads, 1) cluster_decode_kernel(const __grid_constant__ CParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    CCtl& C = *reinterpret_cast<CCtl*>(smem);
    uint8_t* data = smem + (sizeof(CCtl) + 127) / 128 * 128;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = P.H, E = P.E, k = P.k, F = P.F, S = P.S, T = P.T;
    const int n_ent = T * k;
    const bool x_f32 = P.x_dtype != QS_BF16;
    const int rank = (int)cl_rank(), cid = (int)cl_id();
    const int G = P.NCL * kCS;
    const int ns = P.ns;
    uint32_t* status = P.status;
    uint8_t* xraw = data + P.off_x;                                    // [T x H] as given; later hs fp32 [T x S]
    float* hsf = reinterpret_cast<float*>(data + P.off_x);
    const uint8_t* sigbuf = data + P.off_sig;                          // [H] bf16
    uint32_t* xqf = reinterpret_cast<uint32_t*>(data + P.off_xq);      // [T][H/64][36] int16 x fragments
    float* hbuf0 = reinterpret_cast<float*>(data + P.off_hbuf);        // 2 x [T x F] h of a unit's entries
    float* uraw = reinterpret_cast<float*>(data + P.off_uraw);         // [T x F/8] up sums of this CTA's slice
    uint32_t* hqf = reinterpret_cast<uint32_t*>(data + P.off_hq);      // [T][F/64][36] int16 h fragments
    uint8_t* stages = data + P.off_stages;

    if (tid == 0) {
        for (int i = 0; i < ns; i++) {
            mbar_init(&C.full[i], 1);
            mbar_init(&C.empty[i], kCW);
        }
        mbar_init(&C.xbar, 1);
        mbar_init(&C.routed_bar, 1);
        mbar_init(&C.hx[0], kCS);
        mbar_init(&C.hx[1], kCS);
        C.abort = C.issued = C.n_act = C.last = 0;
        C.pub = C.n_ent = 0;
        C.target_g = C.target_t = 0;
        fence_barrier_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();  // every CTA's barriers initialised before any peer touches them
    if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kCW) {
        producer(C, P, data);
        cluster_wait();    // the init phase (a thread waits for a phase before it arrives again)
        cluster_arrive();  // the exit phase: this warp sends nothing to a peer
    } else {
        const Statics st = make_statics(P, blockIdx.x, cid, rank);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (tid == 0) {
            // every earlier call has left; none of this call leaves before every CTA has read this
            const uint64_t n = ld_relaxed_u64(cx_ctr(P, kCxExit)) / (uint64_t)G;
            C.target_g = (n + 1) * (uint64_t)G;
            C.target_t = (n + 1) * (uint64_t)P.NCL;
        }
        int seq = 0;  // stages consumed (its parity picks the partial-sum buffer of a dense stage)
        Ring rg{0, 0u};
        // A stage is handed back only once its copy has landed (after a failed wait it is not:
        // the producer, which watches the abort flag, stops issuing).
        auto stage_wait = [&]() { return warp_wait(C, &C.full[rg.slot], rg.ph, status, 0); };
        auto stage_done = [&](bool landed) {
            __syncwarp();
            if (landed && lane == 0) mbar_arrive(&C.empty[rg.slot]);
            rg.next(ns);
        };
        auto stage_ptr = [&]() { return stages + (size_t)rg.slot * kSB; };
        if (P.x_sys) {  // x from mapped host memory: every load in flight, then the stores
            const int nv = T * H * (x_f32 ? 4 : 2) / 16;
            const uint4* src = static_cast<const uint4*>(P.x);
            uint4* dst = reinterpret_cast<uint4*>(xraw);
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
            cons_sync();
        }
        bool ok = warp_wait(C, &C.xbar, 0, status, 0);

        // ---------------------------------------------------------- x: scales, sigmoid gates, int16 fragments
        {
            // per token (one warp each): max |x| and the shared expert's gate w_sg . x
            if (ok) {
#pragma unroll 1
                for (int t = warp; t < T; t += kCW) {
                    float m = 0.0f, z = 0.0f;
#pragma unroll 2
                    for (int i = lane * 8; i < H; i += 256) {
                        float xv[8], sv[8];
                        load8(xraw + ((size_t)t * H + i) * (x_f32 ? 4 : 2), x_f32, xv);
                        if (S > 0) load8(sigbuf + (size_t)i * 2, false, sv);
#pragma unroll
                        for (int q = 0; q < 8; q++) {
                            m = fmaxf(m, fabsf(xv[q]));
                            if (S > 0) z = fmaf(sv[q], xv[q], z);
                        }
                    }
                    m = warp_max(m);
                    z = warp_sum(z);
                    if (lane == 0) {
                        C.xscale[t] = m;
                        C.gate_s[t] = sigmoid(z);
                    }
                }
            }
            cons_sync();
            if (ok) {
#pragma unroll 1
                for (int i0 = tid * 8; i0 < ((T * H + 255) / 256) * 256; i0 += kCT * 8) {
                    const bool live = i0 < T * H;
                    const int t = live ? i0 >> P.lgH : 0, p = live ? i0 & (H - 1) : 0;
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
                    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                    if (live) {
                        int word, half;
                        frag_pos(p, word, half);
                        uint32_t* row = xqf + (size_t)t * (H / 64) * kFragWords;
                        *reinterpret_cast<uint4*>(row + word) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                        if ((p & 15) == 0) row[(word / kFragWords) * kFragWords + 32 + ((p >> 5) & 3)] = (uint32_t)sum;
                    }
                }
            }
        }

        // ---------------------------------------------------------- router rows -> logits
#pragma unroll 1
        for (int i = 0; i < st.nr; i++, seq++) {
            float(*part)[kMaxT] = C.part[seq & 1];
            const Job j = static_job(P, st, i);
            int nseg = 1;
            if (ok) ok = stage_wait();
            if (ok) nseg = stage_dense<MAXT>(stage_ptr(), true, H, j.n, xraw, x_f32, T, part);
            stage_done(ok);
            cons_sync();
            if (ok) {
#pragma unroll 1
                for (int q = tid; q < j.n * kMaxT; q += kCT) {
                    const int r = q >> 3, t = q & 7, e = j.r0 + r;
                    if (t < T) P.logits[(size_t)t * E + e] = row_dot(part, r, t, nseg) + (P.bias ? P.bias[e] : 0.0f);
                }
            }
        }
        cons_sync();  // orders every logit this CTA stored before the release below
        if (tid == 0) {
            if (!vload(&C.abort)) {
                red_release_add_u64(cx_ctr(P, kCxLogits), 1);
                C.pub |= kPubLogits;
            }
        }
        // ---------------------------------------------------------- routing (every CTA, identically)
        if (tid == 0) {
            const bool got = !vload(&C.abort) && wait_count(cx_ctr(P, kCxLogits), C.target_g, &C.abort);
            if (!got) fail(C, status);
        }
        cons_sync();
        ok = !vload(&C.abort);
        if (ok) {
#pragma unroll 1
            for (int t = warp; t < T; t += kCW) {
                int id;
                float w;
                if (E <= 256) warp_topk<8>(P.logits + (size_t)t * E, E, k, id, w);
                else warp_topk_stream(P.logits + (size_t)t * E, E, k, id, w);
                if (lane < k) {
                    C.ids[t * k + lane] = id;
                    C.p[t * k + lane] = w;
                }
            }
        }
        cons_sync();
        if (ok && warp == 0) {
            // entries ordered by (expert, entry); active experts where the expert changes
#pragma unroll 1
            for (int i = lane; i < n_ent; i += 32) {
                const int e = C.ids[i];
                int r = 0;
#pragma unroll 4
                for (int j = 0; j < n_ent; j++) {
                    const int f = C.ids[j];
                    r += (f < e) | ((f == e) & (j < i));
                }
                C.ent_sorted[r] = i;
                C.es_tok[r] = i / k;
            }
            __syncwarp();
            int na = 0;
#pragma unroll 1
            for (int i0 = 0; i0 < n_ent; i0 += 32) {
                const int i = i0 + lane;
                const bool live = i < n_ent;
                const int e = live ? C.ids[C.ent_sorted[i]] : -1;
                const bool start = live && (i == 0 || C.ids[C.ent_sorted[i - 1]] != e);
                const unsigned bal = __ballot_sync(0xffffffffu, start);
                if (start) {
                    const int a = na + __popc(bal & ((1u << lane) - 1u));
                    C.act_e[a] = e;
                    C.act_begin[a] = i;
                }
                na += __popc(bal);
            }
            if (lane == 0) {
                C.act_begin[na] = n_ent;
                C.n_act = na;
            }
            if (blockIdx.x == 0) {  // the call's routing, for the caller to read back
                for (int i = lane; i < n_ent; i += 32) {
                    P.rec_ids[i] = C.ids[i];
                    P.rec_p[i] = C.p[i];
                }
            }
            __syncwarp();
            __threadfence_block();
            if (lane == 0) mbar_arrive(&C.routed_bar);
        }
        cons_sync();  // the routing tables are read by every warp below
        // ---------------------------------------------------------- shared gate/up rows -> hs
#pragma unroll 1
        for (int i = st.nr; i < st.nr + st.nsg; i++, seq++) {
            // the stage holds j.n gate rows, then the same j.n up rows
            float(*part)[kMaxT] = C.part[seq & 1];
            const Job j = static_job(P, st, i);
            int nseg = 1;
            if (ok) ok = stage_wait();
            if (ok) nseg = stage_dense<MAXT>(stage_ptr(), false, H, 2 * j.n, xraw, x_f32, T, part);
            stage_done(ok);
            cons_sync();
            if (ok) {
#pragma unroll 1
                for (int q = tid; q < j.n * kMaxT; q += kCT) {
                    const int r = q >> 3, t = q & 7;
                    if (t < T)
                        P.hs[(size_t)t * S + j.r0 + r] = silu(row_dot(part, r, t, nseg)) * row_dot(part, j.n + r, t, nseg);
                }
            }
        }
        cons_sync();
        if (tid == 0 && S > 0 && !vload(&C.abort)) {
            red_release_add_u64(cx_ctr(P, kCxHs), 1);
            C.pub |= kPubHs;
        }

        // ---------------------------------------------------------- the cluster's routed experts
        cluster_wait();  // the init phase: every peer's barriers exist
        const int na = C.n_act;  // written before the last consumer barrier: the same in every warp
        const int rowH = P.rowH, rowF = P.rowF, cpr = P.cpr, cpf = P.cpf, PR = P.PR, HS = P.HS;
        // gate/up lane roles: gsz lanes per row (a lane takes chunks c0, c0 + gsz, ...), rpw rows a pass
        const int gsz = P.gsz, grl = lane / gsz, gc0 = lane & (gsz - 1);
        const unsigned ggm = gsz == 32 ? 0xffffffffu : (((1u << gsz) - 1u) << (lane & ~(gsz - 1)));
        // down lane roles: cpf lanes per row, each one chunk
        const int drl = lane / cpf, dc0 = lane & (cpf - 1);
        const unsigned dgm = cpf == 32 ? 0xffffffffu : (((1u << cpf) - 1u) << (lane & ~(cpf - 1)));
        const int dbb = dc0 >> 2, duu = dc0 & 3;
        int ui = 0;
#pragma unroll 1
        for (int u = cid; u < na; u += P.NCL, ui++) {
            const int b = ui & 1;
            float* hb = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(hbuf0) + (size_t)b * P.hbuf_bytes);
            const int jb = C.act_begin[u], nu = C.act_begin[u + 1] - jb;  // the unit's entries
            // one token: its x fragment for this lane's chunk stays in registers for every row
            XFrag fx;
            if (kHoistX && MAXT == 1 && cpr <= 32) load_xfrag_f(xqf + (size_t)gc0 * kFragWords, fx);
            // gate/up rows -> this CTA's slice of h (local)
            int r0g = rank * PR;  // first row of the stage
#pragma unroll 1
            for (int i = 0; i < st.ngu; i++, seq++) {
                const int n = min(P.gp, (rank + 1) * PR - r0g);
                if (ok) ok = stage_wait();
                if (ok) {
                    const uint8_t* sg = stage_ptr();
                    const uint8_t* su = sg + (size_t)n * rowH;
#pragma unroll 1
                    for (int rr = warp * P.rpw; rr < n; rr += kCW * P.rpw) {
                        const int r = rr + grl;
                        const bool live = r < n;
                        const uint8_t* grow = sg + (size_t)r * rowH;
                        const uint8_t* urow = su + (size_t)r * rowH;
                        if (kHoistX && MAXT == 1 && cpr <= 32) {
                            float gv = 0.0f, uv = 0.0f;
                            if (live) {
                                const int boff = (gc0 >> 2) * kBlockBytes;
                                gv = q2k_chunk_dot(grow + boff, gc0 & 3, fx);
                                uv = q2k_chunk_dot(urow + boff, gc0 & 3, fx);
                            }
                            for (int o = gsz >> 1; o > 0; o >>= 1) {
                                gv += __shfl_xor_sync(ggm, gv, o);
                                uv += __shfl_xor_sync(ggm, uv, o);
                            }
                            if (live && gc0 == 0) {
                                const float sx = C.xscale[0] * (1.0f / 32767.0f);
                                hb[r0g + r] = gv * sx;
                                uraw[r0g - rank * PR + r] = uv * sx;
                            }
                        } else {
#pragma unroll 1
                            for (int q = 0; q < nu; q++) {
                                const int t = C.es_tok[jb + q];
                                float gv = 0.0f, uv = 0.0f;
                                if (live) {
#pragma unroll 1
                                    for (int c = gc0; c < cpr; c += gsz) {
                                        XFrag f;
                                        load_xfrag_f(xqf + ((size_t)t * cpr + c) * kFragWords, f);
                                        const int boff = (c >> 2) * kBlockBytes;
                                        gv += q2k_chunk_dot(grow + boff, c & 3, f);
                                        uv += q2k_chunk_dot(urow + boff, c & 3, f);
                                    }
                                }
                                for (int o = gsz >> 1; o > 0; o >>= 1) {
                                    gv += __shfl_xor_sync(ggm, gv, o);
                                    uv += __shfl_xor_sync(ggm, uv, o);
                                }
                                if (live && gc0 == 0) {
                                    const float sx = C.xscale[t] * (1.0f / 32767.0f);
                                    hb[(size_t)q * F + r0g + r] = gv * sx;
                                    uraw[q * PR + r0g - rank * PR + r] = uv * sx;
                                }
                            }
                        }
                    }
                }
                stage_done(ok);
                r0g += P.gp;
            }
            // h = silu(gate) * up over this CTA's slice, four values a thread
            cons_sync();
            const int per = PR >> 2;  // float4s of one entry's slice
            if (ok) {
#pragma unroll 1
                for (int i = tid; i < nu * per; i += kCT) {
                    const int q = i >> P.lgper, v = i & (per - 1);
                    float4* gp4 = reinterpret_cast<float4*>(hb + q * F + rank * PR + 4 * v);
                    const float4 g = *gp4, uu = *reinterpret_cast<const float4*>(uraw + q * PR + 4 * v);
                    *gp4 = make_float4(silu(g.x) * uu.x, silu(g.y) * uu.y, silu(g.z) * uu.z, silu(g.w) * uu.w);
                }
            }
            // this CTA's slice of h to every peer (a thread that stored fences its stores at
            // cluster scope), then one arrival on each peer's barrier, one lane per peer.
            // Thread -> (peer, float4 of the slice); it copies that float4 of every entry.
            cons_sync();
            const bool sender = ok && tid < (kCS - 1) * per;
            if (sender) {
                const int pr = tid >> P.lgper, v = tid & (per - 1);
                const uint32_t peer = (uint32_t)(pr < rank ? pr : pr + 1);
                const uint32_t hl = smem_u32(hb);
#pragma unroll 1
                for (int q = 0; q < nu; q++) {
                    const int off = q * F + rank * PR + 4 * v;
                    st_cluster_v4(cl_map(hl + (uint32_t)off * 4u, peer), *reinterpret_cast<const float4*>(hb + off));
                }
                fence_cluster();
            }
            cons_sync();
            if (warp == 0 && lane < kCS) mbar_arrive_remote(cl_map(smem_u32(&C.hx[b]), (uint32_t)lane));
            // every slice of h: per entry, max-abs int16 fragments
            if (ok) ok = warp_wait(C, &C.hx[b], (ui >> 1) & 1, status, 1);
            if (ok) {
#pragma unroll 1
                for (int q = warp; q < nu; q += kCW) {
                    const float* hr = hb + (size_t)q * F;
                    float m = 0.0f;
#pragma unroll 2
                    for (int p = lane * 8; p < F; p += 256) {
                        const float4 a = *reinterpret_cast<const float4*>(hr + p);
                        const float4 c4 = *reinterpret_cast<const float4*>(hr + p + 4);
                        m = fmaxf(m, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
                        m = fmaxf(m, fmaxf(fmaxf(fabsf(c4.x), fabsf(c4.y)), fmaxf(fabsf(c4.z), fabsf(c4.w))));
                    }
                    m = warp_max(m);
                    const float inv = m > 0.0f ? 32767.0f / m : 0.0f;
                    uint32_t* row = hqf + (size_t)q * cpf * kFragWords;
#pragma unroll 2
                    for (int p = lane * 8; p < F; p += 256) {
                        const float4 a = *reinterpret_cast<const float4*>(hr + p);
                        const float4 c4 = *reinterpret_cast<const float4*>(hr + p + 4);
                        const float hv[8] = {a.x, a.y, a.z, a.w, c4.x, c4.y, c4.z, c4.w};
                        uint32_t wq[4];
                        int sum = 0;
#pragma unroll
                        for (int z = 0; z < 4; z++) {
                            const int a0 = __float2int_rn(hv[2 * z] * inv);
                            const int a1 = __float2int_rn(hv[2 * z + 1] * inv);
                            wq[z] = (uint32_t)(a0 & 0xffff) | ((uint32_t)a1 << 16);
                            sum += a0 + a1;
                        }
                        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                        int word, half;
                        frag_pos(p, word, half);
                        *reinterpret_cast<uint4*>(row + word) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                        if ((p & 15) == 0) row[(word / kFragWords) * kFragWords + 32 + ((p >> 5) & 3)] = (uint32_t)sum;
                    }
                    if (lane == 0) C.hscale[q] = m * (1.0f / 32767.0f);
                }
            }
            cons_sync();
            // one token: its h fragment for this lane's chunk stays in registers for every row
            XFrag fh;
            if (kHoistH && MAXT == 1) load_xfrag_f(hqf + (size_t)dc0 * kFragWords, fh);
            // down rows of slice `rank` -> pd
            int r0d = rank * HS;
#pragma unroll 1
            for (int i = 0; i < st.ndn; i++, seq++) {
                const int n = min(P.dr, (rank + 1) * HS - r0d);
                if (ok) ok = stage_wait();
                if (ok) {
                    const uint8_t* dw = stage_ptr();
#pragma unroll 1
                    for (int rr = warp * P.drpw; rr < n; rr += kCW * P.drpw) {
                        const int r = rr + drl;
                        const bool live = r < n;
                        Q2Chunk cw{};
                        if (live) load_q2chunk(dw + (size_t)r * rowF + dbb * kBlockBytes, duu, cw);
                        if (kHoistH && MAXT == 1) {
                            float v = live ? q2k_chunk_dot(cw, duu, fh) : 0.0f;
                            for (int o = cpf >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(dgm, v, o);
                            if (live && dc0 == 0) P.pd[(size_t)C.ent_sorted[jb] * H + r0d + r] = v * C.hscale[0];
                        } else {
#pragma unroll 1
                            for (int q = 0; q < nu; q++) {
                                float v = 0.0f;
                                if (live) {
                                    XFrag f;
                                    load_xfrag_f(hqf + ((size_t)q * cpf + dc0) * kFragWords, f);
                                    v = q2k_chunk_dot(cw, duu, f);
                                }
                                for (int o = cpf >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(dgm, v, o);
                                if (live && dc0 == 0) P.pd[(size_t)C.ent_sorted[jb + q] * H + r0d + r] = v * C.hscale[q];
                            }
                        }
                    }
                }
                stage_done(ok);
                r0d += P.dr;
            }
        }

        // The exit phase: this CTA sends nothing more to a peer, and every peer's stores and
        // arrivals addressed to it precede the peer's arrival here (release), so once the
        // phase completes no CTA of the cluster can still be written by another.  Arriving
        // now, not at the end, keeps the peers from waiting for this CTA's tail work.
        cluster_arrive();
        // ---------------------------------------------------------- hs -> shared down rows of slice `rank`
        if (S > 0) {
            if (tid == 0 && ok) {
                const bool got = wait_count(cx_ctr(P, kCxHs), C.target_g, &C.abort);
                if (!got) fail(C, status);
            }
            cons_sync();  // also: every warp is done with x long since (hs overwrites it)
            ok = !vload(&C.abort);
            if (ok && st.nsd > 0) {
#pragma unroll 1
                for (int i0 = tid * 4; i0 < T * S; i0 += kCT * 16) {
                    float4 v[4];
#pragma unroll
                    for (int z = 0; z < 4; z++)
                        if (i0 + z * kCT * 4 < T * S) v[z] = ld_relaxed_f32x4(P.hs + i0 + z * kCT * 4);
#pragma unroll
                    for (int z = 0; z < 4; z++)
                        if (i0 + z * kCT * 4 < T * S) *reinterpret_cast<float4*>(hsf + i0 + z * kCT * 4) = v[z];
                }
            }
            cons_sync();
#pragma unroll 1
            for (int i = 0; i < st.nsd; i++, seq++) {
                float(*part)[kMaxT] = C.part[seq & 1];
                const Job j = shared_down_job(P, st, i);
                int nseg = 1;
                if (ok) ok = stage_wait();
                if (ok)
                    nseg = stage_dense<MAXT>(stage_ptr(), false, S, j.n, reinterpret_cast<const uint8_t*>(hsf), true,
                                             T, part);
                stage_done(ok);
                cons_sync();
                if (ok) {
#pragma unroll 1
                    for (int q = tid; q < j.n * kMaxT; q += kCT) {
                        const int r = q >> 3, t = q & 7;
                        if (t < T) P.sdp[(size_t)t * H + j.r0 + r] = row_dot(part, r, t, nseg);
                    }
                }
            }
        }

        // ---------------------------------------------------------- slice ticket; the last CTA sums
        cons_sync();  // orders this CTA's pd / sdp stores before the ticket
        if (tid == 0) {
            int last = 0;
            __threadfence();
            const uint64_t old = atom_add_acq_rel_u64(cx_ctr(P, kCxTicket + rank), 1);
            C.pub |= kPubTicket;
            if (!vload(&C.abort) && old + 1 == C.target_t) last = 1;
            C.last = last;
        }
        cons_sync();
        if (C.last && !vload(&C.abort)) {
            const int r0 = rank * HS;
#pragma unroll 1
            for (int i = tid; i < T * HS; i += kCT) {
                const int t = i / HS, r = r0 + i % HS;
                float v[33];
#pragma unroll
                for (int j = 0; j < 32; j++)  // every load in flight before the first is used
                    if (j < k) v[j] = ld_relaxed_f32(P.pd + (size_t)(t * k + j) * H + r);
                v[32] = S > 0 ? ld_relaxed_f32(P.sdp + (size_t)t * H + r) : 0.0f;
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; j++)
                    if (j < k) acc = fmaf(C.p[t * k + j], v[j], acc);
                if (S > 0) acc = fmaf(C.gate_s[t], v[32], acc);
                P.out[(size_t)t * H + r] = acc;
            }
        }
    }

    // ---------------------------------------------------------- wind-down
    __syncthreads();
    if (tid == 0) {
        // never leave a copy in flight into shared memory that is about to be released
        const int issued = vload(&C.issued);
#pragma unroll 1
        for (int s = max(0, issued - ns); s < issued; s++)
            if (!mbar_wait(&C.full[s % ns], (s / ns) & 1)) set_status(status, QS_ERR_TIMEOUT);
        if (!mbar_wait(&C.xbar, 0)) set_status(status, QS_ERR_TIMEOUT);
        if (vload(&C.abort)) set_status(status, QS_ERR_TIMEOUT);
        // keep every counter at its per-call increment, whatever happened
        const int pub = vload(&C.pub);
        if (!(pub & kPubLogits)) red_relaxed_add_u64(cx_ctr(P, kCxLogits), 1);
        if (!(pub & kPubHs)) red_relaxed_add_u64(cx_ctr(P, kCxHs), 1);
        if (!(pub & kPubTicket)) red_relaxed_add_u64(cx_ctr(P, kCxTicket + rank), 1);
        red_relaxed_add_u64(cx_ctr(P, kCxExit), 1);
    }
    // no CTA leaves while a peer may still write its shared memory or arrive on its barriers
    cluster_wait();
}

// ------------------------------------------------------------------ host side

size_t up16(size_t v) { return (v + 15) / 16 * 16; }
bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

struct CPlanHost {
    int ns, rr, ps, dsr, gp, dr;
    int off_x, off_sig, off_xq, off_hbuf, off_hq, off_uraw, off_stages, hbuf_bytes;
    size_t smem;
};

bool plan_cluster(const qs_moe_shape& s, int T, size_t smem_max, CPlanHost& cp) {
    const int H = s.hidden, E = s.n_experts, k = s.top_k, F = s.expert_ffn, S = s.shared_ffn;
    const int nbH = H / 256, nbF = F / 256;
    const int xsz = s.x_dtype == QS_BF16 ? 2 : 4;
    if (T < 1 || T > kMaxT || T * k > kMaxEnt || k > 32 || E > 1024) return false;
    if (!pow2(nbH) || nbH > 32 || !pow2(nbF) || 4 * nbF > 32) return false;
    if (H * 4 > kSB || (S > 0 && (4 * H > kSB || 2 * S > kSB))) return false;
    const int PR = F / kCS, HS = H / kCS;
    if (F % (4 * kCS) || H % (4 * kCS)) return false;  // 16-byte aligned row spans of every CTA
    const int rowH = nbH * 84, rowF = nbF * 84;
    cp.rr = std::max(1, kSB / (H * 4));
    cp.ps = S > 0 ? kSB / (4 * H) : 1;
    cp.dsr = S > 0 ? kSB / (2 * S) : 1;
    {
        // routed gate/up pairs a stage: a whole number of warp passes when the stage holds more
        const int cpr = H / 64, rpw = 32 / std::min(cpr, 32);
        int gp = std::min(PR, kSB / (2 * rowH));
        if (gp >= kCW * rpw) gp = gp / (kCW * rpw) * (kCW * rpw);
        while (gp > 0 && ((size_t)gp * rowH) % 16) gp--;  // 16-byte bulk copies
        cp.gp = gp;
    }
    cp.dr = std::min(HS, kSB / rowF) / 4 * 4;
    if (cp.gp < 1 || cp.dr < 4) return false;
    size_t o = 0;
    cp.off_x = (int)o;
    o += up16(std::max((size_t)T * H * xsz, (size_t)T * S * 4));
    cp.off_sig = (int)o;
    o += up16((size_t)H * 2);
    cp.off_xq = (int)o;
    o += (size_t)T * (H / 64) * kFragWords * 4;
    cp.hbuf_bytes = (int)up16((size_t)T * F * 4);
    cp.off_hbuf = (int)o;
    o += 2 * (size_t)cp.hbuf_bytes;
    cp.off_hq = (int)o;
    o += (size_t)T * (F / 64) * kFragWords * 4;
    cp.off_uraw = (int)o;
    o += up16((size_t)T * PR * 4);
    o = (o + 127) / 128 * 128;
    cp.off_stages = (int)o;
    const size_t fixed = (sizeof(CCtl) + 127) / 128 * 128 + o;
    if (fixed + 3 * (size_t)kSB > smem_max) return false;
    cp.ns = (int)std::min<size_t>(kMaxNS, (smem_max - fixed) / kSB);
    cp.smem = fixed + (size_t)cp.ns * kSB;
    return true;
}

struct CFacts {
    int n_sm = 0, smem_max = 0;
    int ncl[4] = {0, 0, 0, 0};  // clusters co-resident per instantiation (0 = not queried yet)
};
constexpr int kMaxDevices = 64;
CFacts g_cf[kMaxDevices];
std::mutex g_cf_mutex;

cudaError_t cfacts(CFacts** out, int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    CFacts& f = g_cf[dev];
    if (f.n_sm == 0) {
        int n = 0, m = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        f.smem_max = m;
        f.n_sm = n;
    }
    *out = &f;
    *dev_out = dev;
    return cudaSuccess;
}

template <int MAXT>
void* kernel_fn() {
    return (void*)cluster_decode_kernel<MAXT>;
}

int slot_of(int T) { return T == 1 ? 0 : T <= 2 ? 1 : T <= 4 ? 2 : 3; }

// Clusters of kCS CTAs that fit at once with `smem` bytes each (cached per instantiation; the
// largest plan of any call sets the shared-memory limit once).
template <int MAXT>
cudaError_t clusters_for(CFacts& f, int slot, int* ncl) {
    std::lock_guard<std::mutex> lock(g_cf_mutex);
    if (f.ncl[slot] == 0) {
        const void* fn = kernel_fn<MAXT>();
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, f.smem_max);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = kCS;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(kCS);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = (size_t)f.smem_max;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, cluster_decode_kernel<MAXT>, &cfg);
        if (e != cudaSuccess) return e;
        f.ncl[slot] = n > 0 ? std::min(n, f.n_sm / kCS) : -1;
    }
    *ncl = f.ncl[slot];
    return cudaSuccess;
}

template <int MAXT>
cudaError_t launch_t(CParams& p, size_t smem, CFacts& f, int slot, cudaStream_t st) {
    int ncl = 0;
    cudaError_t e = clusters_for<MAXT>(f, slot, &ncl);
    if (e != cudaSuccess) return e;
    if (ncl < 1) return cudaErrorNotSupported;
    p.NCL = ncl;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kCS;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(ncl * kCS);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, cluster_decode_kernel<MAXT>, p);
}

}  // namespace

bool cluster_decode_supported(const qs_moe_shape& s, int T, cudaError_t* err) {
    CFacts* f = nullptr;
    int dev = 0;
    *err = cfacts(&f, &dev);
    if (*err != cudaSuccess) return false;
    CPlanHost cp;
    if (!plan_cluster(s, T, (size_t)f->smem_max, cp)) return false;
    int ncl = 0;  // and whether its clusters fit on this device at all
    const int slot = slot_of(T);
    *err = T == 1 ? clusters_for<1>(*f, slot, &ncl)
         : T <= 2 ? clusters_for<2>(*f, slot, &ncl)
         : T <= 4 ? clusters_for<4>(*f, slot, &ncl)
                  : clusters_for<8>(*f, slot, &ncl);
    return *err == cudaSuccess && ncl >= 1;
}

cudaError_t launch_cluster_decode(const qs_moe_shape& s, const void* x, const float* Wr, const float* bias,
                                  const uint8_t* experts, int64_t stride, const uint16_t* sg, const uint16_t* su,
                                  const uint16_t* sd, const uint16_t* ssig, int T, float* out, void* ws,
                                  const WsLayout& W, cudaStream_t st, bool x_host_mapped) {
    CFacts* f = nullptr;
    int dev = 0;
    cudaError_t e = cfacts(&f, &dev);
    if (e != cudaSuccess) return e;
    qs_moe_shape eff = s;
    if (sg == nullptr) eff.shared_ffn = 0;
    CPlanHost cp;
    if (!plan_cluster(eff, T, (size_t)f->smem_max, cp)) return cudaErrorNotSupported;
    CParams p;
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
    p.logits = reinterpret_cast<float*>(base + W.xlog);
    p.hs = reinterpret_cast<float*>(base + W.xhs);
    p.pd = reinterpret_cast<float*>(base + W.cpd);
    p.sdp = reinterpret_cast<float*>(base + W.csdp);
    p.rec_ids = reinterpret_cast<int32_t*>(base + W.ids);
    p.rec_p = reinterpret_cast<float*>(base + W.pw);
    p.cx = base + W.cx;
    p.status = reinterpret_cast<uint32_t*>(base + W.header);
    p.H = eff.hidden;
    p.E = eff.n_experts;
    p.k = eff.top_k;
    p.F = eff.expert_ffn;
    p.S = eff.shared_ffn;
    p.T = T;
    p.x_dtype = eff.x_dtype;
    p.x_sys = x_host_mapped ? 1 : 0;
    p.NCL = 0;
    p.ns = cp.ns;
    p.rr = cp.rr;
    p.ps = cp.ps;
    p.dsr = cp.dsr;
    p.gp = cp.gp;
    p.dr = cp.dr;
    p.off_x = cp.off_x;
    p.off_sig = cp.off_sig;
    p.off_xq = cp.off_xq;
    p.off_hbuf = cp.off_hbuf;
    p.off_hq = cp.off_hq;
    p.off_uraw = cp.off_uraw;
    p.off_stages = cp.off_stages;
    p.hbuf_bytes = cp.hbuf_bytes;
    {
        const int H = eff.hidden, F = eff.expert_ffn;
        p.lgH = 0;
        while ((1 << p.lgH) < H) p.lgH++;
        p.rowH = H / 256 * kBlockBytes;
        p.rowF = F / 256 * kBlockBytes;
        p.cpr = H / 64;
        p.cpf = F / 64;
        p.gsz = std::min(p.cpr, 32);
        p.rpw = 32 / p.gsz;
        p.drpw = 32 / p.cpf;
        p.PR = F / kCS;
        p.HS = H / kCS;
        p.lgper = 0;
        while ((1 << p.lgper) < p.PR / 4) p.lgper++;
    }
    const int slot = slot_of(T);
    if (T == 1) return launch_t<1>(p, cp.smem, *f, slot, st);
    if (T <= 2) return launch_t<2>(p, cp.smem, *f, slot, st);
    if (T <= 4) return launch_t<4>(p, cp.smem, *f, slot, st);
    return launch_t<8>(p, cp.smem, *f, slot, st);
}

}  // namespace qs

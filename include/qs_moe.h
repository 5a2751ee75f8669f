/*
 * qs_moe.h -- C ABI of the GB300 (sm_103a) Q2_K mixture-of-experts FFN layer.
 *
 * The layer, per token t with input x_t [H]:
 *   logits  l = W_r x_t (+ b)                       router GEMV, fp32 weights
 *   ids     the top_k largest logits, descending, ties to the lower expert id
 *   p       softmax over the top_k selected logits (sums to 1)
 *   h_j     silu(W_gate[e_j] x_t) * (W_up[e_j] x_t)  routed experts, Q2_K weights
 *   y_t     sum_j p_j W_down[e_j] h_j
 *         + sigmoid(w_sg . x_t) * W_sd (silu(W_sg x_t) * (W_su x_t))   bf16 shared expert
 *
 * Sources: QuarkStar (q36) README, "Model Weights", and DwarfStar (ds4) page,
 * "Model Weights" -- routed experts are 2-bit, shared experts, projections
 * and routing stay in higher precision; Quasar (q27) README, "Architecture
 * facts" (SwiGLU FFN) and "Design decisions" (dequantisation fused into the
 * GEMV); the layer's workload statement (router GEMV + softmax + top-k, Q2_K
 * gate/up/down, sigmoid-gated bf16 shared expert, weighted sum).
 *
 * Q2_K block (256 weights in 84 bytes, GGUF layout as the QuarkStar README,
 * "Acknowledgements", says is retained): scales[16] at bytes 0..15 (low
 * nibble = scale, high nibble = min), qs[64] at bytes 16..79 (weight
 * i = 128h + 32j + l is bits 2j..2j+1 of qs[32h + l]), fp16 d at bytes
 * 80..81 and fp16 dmin at 82..83, little-endian; weight i of the block is
 * d * (scales[i/16] & 15) * q_i - dmin * (scales[i/16] >> 4).
 *
 * Expert blob layout: expert e starts at blocks + e * expert_stride; inside,
 * gate rows [F x H], then up rows [F x H], then down rows [H x F]; each row is
 * K/256 consecutive blocks along its K (contiguous) dimension.
 *
 * Conventions of every entry point:
 *  - Pointers named device are device memory; the caller owns every buffer.
 *    The library allocates nothing (apart from the fixed array behind
 *    qs_moe_ffn_noalloc) and keeps no per-call state; it caches per-device
 *    facts (SM count, shared-memory limit) on first use.
 *  - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL =
 *    the legacy default stream).  Calls on one workspace must not overlap.
 *  - Host-detectable argument errors return QS_ERR_INVALID (or
 *    QS_ERR_WORKSPACE / QS_ERR_UNSUPPORTED) before anything is launched.
 *  - A failed launch returns QS_ERR_CUDA; qs_last_cuda_error() gives the
 *    cudaError_t of the calling thread's last failure.
 *  - Device-side failures (a bounded wait that ran out) are recorded in a
 *    sticky status word in the workspace and read with qs_read_device_status.
 *  - Requirements: hidden % 256 == 0, expert_ffn % 256 == 0, shared_ffn %
 *    256 == 0 (or 0 = no shared expert), hidden and expert_ffn <= 8192,
 *    1 <= top_k <= min(n_experts, 32), n_experts <= 1024, n_tokens >= 1,
 *    the workspace 256-byte aligned, the expert blob base and
 *    expert_stride 16-byte aligned, x and every bf16 matrix 16-byte aligned.
 */
#ifndef QS_MOE_H_
#define QS_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

#define QS_ABI_VERSION 1

typedef enum {
    QS_OK = 0,
    QS_ERR_INVALID = 1,      /* bad argument (null, shape, alignment)            */
    QS_ERR_CUDA = 2,         /* a CUDA runtime call or kernel launch failed       */
    QS_ERR_TIMEOUT = 3,      /* a bounded device-side wait ran out (sticky)       */
    QS_ERR_UNSUPPORTED = 4,  /* a valid request this build does not implement     */
    QS_ERR_WORKSPACE = 5     /* workspace missing or smaller than required        */
} qs_status;

typedef enum { QS_F32 = 0, QS_BF16 = 1 } qs_dtype;

/* Layer shape.  x_dtype is the storage type of x (fp32 or bf16). */
typedef struct {
    int32_t hidden;      /* H */
    int32_t n_experts;   /* E */
    int32_t top_k;       /* k */
    int32_t expert_ffn;  /* F */
    int32_t shared_ffn;  /* S, 0 = no shared expert */
    int32_t x_dtype;     /* qs_dtype */
} qs_moe_shape;

/* Routed experts in Q2_K (device memory, read only). */
typedef struct {
    const void *blocks;     /* expert 0's first byte; 16-byte aligned             */
    int64_t expert_stride;  /* bytes between experts, >= the expert's Q2_K bytes, % 16 == 0 */
} qs_q2k_experts;

/* Routed experts in Q4_K (device memory, read only): per expert gate rows
 * [F x H], up rows [F x H], down rows [H x F], 144-byte blocks of 256 weights
 * along each row (GGUF Q4_K layout, which the pages keep: QuarkStar (q36)
 * README, "Acknowledgements"; Q4_K experts: its "Model Weights" section):
 * d (fp16 LE) | dmin (fp16 LE) | 12 bytes of 6-bit scales and mins for eight
 * 32-weight sub-blocks | 128 bytes of 4-bit codes. */
typedef struct {
    const void *blocks;     /* expert 0's first byte; 16-byte aligned             */
    int64_t expert_stride;  /* bytes between experts, >= the expert's Q4_K bytes, % 16 == 0 */
} qs_q4k_experts;

/* bf16 shared expert (device memory, read only, row-major). */
typedef struct {
    const void *w_gate;      /* [S x H] */
    const void *w_up;        /* [S x H] */
    const void *w_down;      /* [H x S] */
    const void *w_gate_sig;  /* [H], the sigmoid gate vector w_sg */
} qs_shared_expert;

/* Static description of a status code (never NULL). */
const char *qs_status_string(int status);

/* QS_ABI_VERSION of the loaded library. */
int qs_abi_version(void);

/* cudaError_t of the calling thread's last QS_ERR_CUDA (0 if none). */
int qs_last_cuda_error(void);

/* Bytes of workspace qs_moe_ffn / qs_route_topk need for up to max_tokens
 * tokens (0 on an invalid shape).  The first 256 bytes are the header: the
 * sticky status word and the counters of the device-side waits. */
size_t qs_moe_workspace_bytes(const qs_moe_shape *shape, int max_tokens);

/* Zero the workspace header (status word and wait counters).  Must run once
 * before the first use of a workspace and after a QS_ERR_TIMEOUT. */
int qs_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/* Synchronise `stream`, then return the sticky device status of the
 * workspace (QS_OK or QS_ERR_TIMEOUT), or QS_ERR_CUDA if the sync failed. */
int qs_read_device_status(const void *workspace, void *stream);

/* (a) Router GEMV + softmax + top-k.
 * x        device [n_tokens x H], shape->x_dtype
 * router_w device fp32 [E x H];  router_bias device fp32 [E] or NULL
 * topk_ids device int32 [n_tokens x k], expert ids in descending-logit order
 * topk_w   device fp32  [n_tokens x k], softmax of the selected logits
 * workspace: qs_moe_workspace_bytes(shape, n_tokens) bytes, initialised.
 * Logits are accumulated in fp32; ties go to the lower expert id. */
int qs_route_topk(const qs_moe_shape *shape, const void *x, const float *router_w, const float *router_bias,
                  int n_tokens, int32_t *topk_ids, float *topk_w, void *workspace, size_t workspace_bytes,
                  void *stream);

/* (b) Token -> expert grouping.
 * topk_ids device int32 [n_tokens x k]; entries outside [0, E) are left
 *          out of every group (then offsets[E] < n_tokens*k)
 * counts   device int32 [E]       tokens routed to each expert
 * offsets  device int32 [E + 1]   exclusive prefix sum of counts
 * perm     device int32 [n_tokens*k] flat entries t*k+slot listed expert by
 *          expert, ascending inside each expert (stable). */
int qs_group_tokens(const qs_moe_shape *shape, const int32_t *topk_ids, int n_tokens, int32_t *counts,
                    int32_t *offsets, int32_t *perm, void *stream);

/* (c) Grouped Q2_K gate+up dequant-GEMV with SwiGLU epilogue.
 * For every entry j of perm (expert e = the group j falls in, token
 * t = perm[j] / k): h_out[perm[j], :] = silu(W_gate[e] x_t) * (W_up[e] x_t).
 * x device [n_tokens x H]; offsets/perm from qs_group_tokens;
 * h_out device fp32 [n_tokens*k x F].  x is quantised per token to int16
 * with a max-abs scale; block dot products are exact in int32, the rest fp32. */
int qs_q2k_gemv_grouped(const qs_moe_shape *shape, const void *x, const qs_q2k_experts *experts,
                        const int32_t *offsets, const int32_t *perm, int n_tokens, float *h_out, void *stream);

/* (d) Q2_K down-projection GEMV with the routing-weight combine.
 * out[t, :] (+)= sum over the token's slots, in ascending expert order, of
 * topk_w[t, slot] * W_down[e] h[t*k + slot, :].
 * topk_ids/topk_w device [n_tokens x k]; h device fp32 [n_tokens*k x F];
 * out device fp32 [n_tokens x H]; accumulate != 0 adds into out. */
int qs_q2k_down_combine(const qs_moe_shape *shape, const qs_q2k_experts *experts, const float *h,
                        const int32_t *topk_ids, const float *topk_w, int n_tokens, float *out, int accumulate,
                        void *stream);

/* Gated bf16 shared expert alone:
 * out[t, :] (+)= sigmoid(w_sg . x_t) * W_sd (silu(W_sg x_t) * (W_su x_t)).
 * workspace: qs_moe_workspace_bytes(shape, n_tokens) bytes. */
int qs_shared_expert_ffn(const qs_moe_shape *shape, const void *x, const qs_shared_expert *shared, int n_tokens,
                         float *out, int accumulate, void *workspace, size_t workspace_bytes, void *stream);

/* The whole layer: out [n_tokens x H] fp32 (overwritten) = routed experts
 * + gated shared expert (shared may be NULL or have S = 0).  workspace:
 * qs_moe_workspace_bytes(shape, n_tokens) bytes, initialised with
 * qs_workspace_init.  Three implementations, picked per call:
 *  - n_tokens <= 16 and a shape the persistent decode kernel plans for: one
 *    kernel of one CTA per SM that needs every SM at once (other work holding
 *    SMs for longer than the wait bound ends the call in QS_ERR_TIMEOUT).  It
 *    is a programmatic dependent launch: it may start while the previous
 *    kernel in the stream finishes, prefetching weights into L2 meanwhile, and
 *    waits for that kernel before it reads x or writes anything.  The result
 *    does not depend on how tokens are batched;
 *  - else, up to 8 tokens, the cluster decode kernel (qs_moe_ffn_cluster);
 *  - otherwise, with bf16 x (and Q2_K rows it can stage: hidden a multiple of
 *    1024 or equal to 256; expert_ffn a multiple of 1024 or at most 768): the
 *    tensor-core path -- router on the tensor cores as three exact bf16 planes
 *    of router_w, experts as grouped GEMMs with Q2_K weights dequantised to
 *    fp16 (the shared expert in bf16), fp32 accumulation, each routed
 *    contribution p * (W_down h) rounded to fp16 and the k of a token summed in
 *    slot order onto the shared expert's fp32 row;
 *  - otherwise the per-step kernels (c)/(d) above. */
int qs_moe_ffn(const qs_moe_shape *shape, const void *x, const float *router_w, const float *router_bias,
               const qs_q2k_experts *experts, const qs_shared_expert *shared, float *out, int n_tokens,
               void *workspace, size_t workspace_bytes, void *stream);

/* The whole layer through the cluster decode kernel alone (no other path):
 * the grid is thread-block clusters of 8 CTAs, one CTA per SM; a cluster owns
 * whole routed experts -- its 8 CTAs each compute 1/8 of an expert's gate/up
 * rows, share the slices of h through distributed shared memory, and each
 * forms the expert's down product over 1/8 of the output rows -- and a
 * per-slice ticket lets the CTA that completes a slice add the experts' down
 * products and the shared expert's in slot order.  Same arguments, result
 * (within the layer's tolerance), workspace and error behaviour as
 * qs_moe_ffn, for up to 8 tokens with top_k * n_tokens <= 64 and
 * power-of-two block counts per row; otherwise QS_ERR_UNSUPPORTED.
 * qs_moe_ffn does not pick it first: measured on GB300 it is slower than the
 * persistent kernel at every token count tried, because with 15 clusters of 8
 * only the clusters that own an active expert carry the routed rows (64 of 120
 * SMs at one token).  Needs every cluster resident at once, like the
 * persistent kernel (a wait bound ends the call in QS_ERR_TIMEOUT otherwise). */
int qs_moe_ffn_cluster(const qs_moe_shape *shape, const void *x, const float *router_w, const float *router_bias,
                       const qs_q2k_experts *experts, const qs_shared_expert *shared, float *out, int n_tokens,
                       void *workspace, size_t workspace_bytes, void *stream);

/* The whole layer without a workspace argument (the pages have no
 * counterpart; this is a convenience of this library).  For callers that
 * cannot allocate device memory -- an operator inside a framework that owns
 * every device allocation and passes only inputs and outputs, or a serving loop
 * under a fixed memory budget where cudaMalloc is not allowed once it runs.
 * Same arguments and result as qs_moe_ffn minus the workspace; only the
 * persistent decode kernel runs (n_tokens <= 16 and the shapes it plans for),
 * otherwise QS_ERR_UNSUPPORTED.  Its scratch is a fixed 4 MiB array inside the
 * library, held on every GPU that loads it until the process exits; a token
 * count whose exchange area exceeds it returns QS_ERR_WORKSPACE.  The first
 * call on a device looks the array up and zeroes it, synchronising `stream`,
 * so make that first call before any stream capture.  Every call on a device
 * shares the array and it keeps the last call's contents; calls that overlap
 * on the GPU race on it.  A device-side time-out (the persistent kernel waits
 * for every CTA, so other work holding SMs past the wait bound ends it early)
 * leaves out's rows incomplete and is recorded in the array's sticky status
 * word: read it with qs_noalloc_read_device_status after the call. */
int qs_moe_ffn_noalloc(const qs_moe_shape *shape, const void *x, const float *router_w, const float *router_bias,
                       const qs_q2k_experts *experts, const qs_shared_expert *shared, float *out, int n_tokens,
                       void *stream);

/* Synchronise `stream`, then return the sticky device status of the current
 * device's qs_moe_ffn_noalloc array (QS_OK, or QS_ERR_TIMEOUT if a call since
 * the last read ran out of a device-side wait and its output is not valid) and
 * clear it.  QS_OK if no qs_moe_ffn_noalloc call has run on this device;
 * QS_ERR_CUDA if the sync or the 4-byte copies fail.  Allocates nothing. */
int qs_noalloc_read_device_status(void *stream);

/* The whole layer with Q4_K routed experts: the same routing, grouping and
 * gated bf16 shared expert as qs_moe_ffn, the routed gate/up (SwiGLU) and down
 * projections dequantising Q4_K blocks (w = d*sc*q - dmin*m per 32-weight
 * sub-block).  Arguments, layouts, workspace (qs_moe_workspace_bytes of the
 * same shape) and error behaviour as qs_moe_ffn; expert_stride must cover
 * 144*3*F*H/256 bytes and be a multiple of 16.  Where the persistent decode
 * kernel plans the call (the token counts it takes for qs_moe_ffn) it is one
 * launch: activations quantised per token to int16 with a max-abs scale,
 * per-chunk integer sums exact, d and dmin applied in fp32.  Otherwise the
 * per-step kernels (fp32 activations, fp32 accumulation): up to six launches
 * on `stream`. */
int qs_moe_ffn_q4k(const qs_moe_shape *shape, const void *x, const float *router_w, const float *router_bias,
                   const qs_q4k_experts *experts, const qs_shared_expert *shared, float *out, int n_tokens,
                   void *workspace, size_t workspace_bytes, void *stream);

/* Q4_K encoder (weight set-up, not part of the layer): round-to-nearest, per
 * 32-weight sub-block m = max(0, -min), s = (max + m)/15, per block
 * d = fp16(max s / 63), dmin = fp16(max m / 63), 6-bit scale and min codes and
 * 4-bit weight codes by rint, every decision in fp32.  w device fp32
 * [n_rows x K], K % 256 == 0, 16-byte aligned; out device [n_rows x K/256 x
 * 144] bytes (4-byte aligned). */
int qs_q4k_quantize(const float *w, int64_t n_rows, int64_t K, void *out, void *stream);

/* Directional steering of the layer's output, in place (QuarkStar (q36)
 * README, "Steering"; DwarfStar (ds4) page, "Steering"): every token row
 * y of out is replaced by y - scale * direction * (direction . y).
 * out: device fp32 [n_tokens x hidden], row-major, the rows a qs_moe_ffn call
 * wrote (or any rows); direction: device fp32 [hidden], the layer's
 * direction as stored (normalised by the caller; the library does not
 * normalise it).  Positive scale removes the direction, negative amplifies
 * it; scale == 0 is the unsteered path and launches nothing.  hidden must be a
 * positive multiple of 4 and both pointers 16-byte aligned; otherwise
 * QS_ERR_INVALID before any launch.  One kernel on `stream`, one CTA per row,
 * the dot product summed in a fixed order (run-to-run identical).  The caller
 * owns both buffers. */
int qs_steer_rows(float *out, const float *direction, float scale, int n_tokens, int hidden, void *stream);

/* The whole layer with x and out in host memory: queues on `stream` a copy of
 * x (host, [n_tokens x H], x_dtype) into the workspace, the qs_moe_ffn call
 * and a copy of the result into out_host (host fp32 [n_tokens x H]), then
 * returns; synchronise the stream before reading out_host.  When both host
 * buffers are pinned (page-locked, so mapped into the device's address space;
 * 16-byte aligned) and the call is one the cluster decode kernel takes, that
 * kernel reads x and writes out through their mapped addresses instead, with
 * no copies queued.  Host buffers should be pinned for the copies to be
 * asynchronous.  Weights,
 * shared expert and workspace are device memory as for qs_moe_ffn;
 * workspace: qs_moe_host_workspace_bytes(shape, n_tokens) bytes, 256-byte
 * aligned, initialised with qs_workspace_init (the layer's workspace first,
 * then the device copies of x and out).  Errors as qs_moe_ffn. */
size_t qs_moe_host_workspace_bytes(const qs_moe_shape *shape, int max_tokens);
int qs_moe_ffn_host(const qs_moe_shape *shape, const void *x_host, const float *router_w, const float *router_bias,
                    const qs_q2k_experts *experts, const qs_shared_expert *shared, float *out_host, int n_tokens,
                    void *workspace, size_t workspace_bytes, void *stream);

/* The routing the last qs_moe_ffn (or qs_moe_ffn_host) call on `workspace`
 * chose, as its kernels used it: synchronise `stream`, then copy to host memory
 * ids_host int32 [n_tokens x k] (expert ids, descending logit, ties to the lower
 * id) and w_host fp32 [n_tokens x k] (softmax over the selected logits).
 * n_tokens and shape must be the call's; workspace as for qs_moe_ffn.  Every
 * implementation records it (the one-kernel paths from their first CTA, after
 * its top-k; the others from their routing kernel).  QS_ERR_CUDA if the sync or
 * a copy fails. */
int qs_read_routing(const qs_moe_shape *shape, int n_tokens, const void *workspace, size_t workspace_bytes,
                    int32_t *ids_host, float *w_host, void *stream);

/* Number of kernels one qs_moe_ffn call with this shape, token count and
 * shared expert (has_shared != 0) launches on the current device: 1 for the
 * persistent decode kernel, 8 for the tensor-core path (which also issues a
 * memset), 4 or 5 for the per-step path; 0 on an invalid shape, negative
 * (-cudaError_t) if the device query fails. */
int qs_moe_ffn_launches(const qs_moe_shape *shape, int n_tokens, int has_shared);

/* The same count for qs_moe_ffn_q4k: 1 for the persistent decode kernel, else
 * 6 (4 without the shared expert); 0 on an invalid shape, negative
 * (-cudaError_t) if the device query fails. */
int qs_moe_ffn_q4k_launches(const qs_moe_shape *shape, int n_tokens, int has_shared);

/* Q2_K encoder (weight set-up, not part of the layer): round-to-nearest,
 * per sub-block m = max(0, -min), s = (max + m)/3, per block d = fp16(max s
 * / 15), dmin = fp16(max m / 15), 4-bit nibbles and 2-bit codes by rint,
 * every decision in fp32.  w device fp32 [n_rows x K], K % 256 == 0;
 * out device [n_rows x K/256 x 84] bytes (4-byte aligned). */
int qs_q2k_quantize(const float *w, int64_t n_rows, int64_t K, void *out, void *stream);

/* Test hook for the bounded device-side wait: launches one CTA that waits
 * on a workspace counter nothing increments, for at most limit_us
 * microseconds (1..1e6); the CTA then records QS_ERR_TIMEOUT in the status
 * word and returns.  Checks that a wait that runs out reports instead of
 * hanging. */
int qs_test_wait_timeout(void *workspace, size_t workspace_bytes, int limit_us, void *stream);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif
#ifdef __cplusplus
}
#endif
#endif /* QS_MOE_H_ */

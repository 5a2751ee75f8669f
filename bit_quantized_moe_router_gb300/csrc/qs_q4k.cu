// qs_q4k.cu -- routed experts in the 4-bit Q4_K super-block format (sm_103a).
//
// The pages name Q4_K experts for the late layers (QuarkStar (q36) README,
// "Model Weights": the Layers34-39Q4KExperts file) and keep GGUF quant
// layouts ("Acknowledgements"); the block is read as GGUF's Q4_K, 144 bytes
// per 256 weights:
//   d (fp16 LE) | dmin (fp16 LE) | scales[12] | qs[128]
// eight 32-weight sub-blocks j with a 6-bit scale and a 6-bit min
//   j < 4:  sc = S[j] & 63,                           m = S[j+4] & 63
//   j >= 4: sc = (S[j+4] & 15) | (S[j-4] >> 6) << 4,  m = (S[j+4] >> 4) | (S[j] >> 6) << 4
// weight 64c + l is the low nibble of qs[32c + l] (l < 32, sub-block 2c) or the
// high nibble of qs[32c + l - 32] (sub-block 2c + 1); w = d * sc * q - dmin * m.
//
// Kernels (the per-step path of the layer with Q4_K experts; routing, grouping
// and the shared expert are the Q2_K path's kernels):
//   q4k_quantize_kernel  fp32 rows -> blocks, one warp per block (set-up step)
//   q4k_gateup_kernel    CTA per (active expert, tile of R rows); the tile's gate
//                        and up rows are staged in shared memory by two bulk
//                        copies; per routed token, its x row (fp32, as float4
//                        groups ordered [group][sub-block], so that a warp's
//                        lanes read consecutive groups) and the sums of x over
//                        each 32-weight sub-block are staged; a warp takes a
//                        row, a lane a sub-block (lanes stride over the row's
//                        sub-blocks), one fixed shuffle reduction
//   q4k_down_kernel      CTA per (tile of 4 or 16 output rows, token); the token's
//                        k rows of h and their sub-block sums are staged; a warp
//                        takes a (row, slot) pair's dot product; one thread per
//                        row sums the k slots' dots, each weighted by its routing
//                        weight, in slot order
// Per 32-weight sub-block the dot is sum(q*x) in fp32 (one FMA per weight after
// the nibble is extracted) and the sub-block result d*sc*sum(q*x) - dmin*m*sum(x).
#include "qs_common.cuh"
#include "qs_internal.h"

#include <algorithm>

namespace qs {

constexpr int kQ4Bytes = 144;

// ====================================================================== encoder

// Round-to-nearest encoder, every decision in fp32 in the order of the oracle's
// encoder (one rounding per operation, ties to even): per sub-block
// m = max(0, -min), s = (max + m) / 15; per block d = fp16(max s / 63),
// dmin = fp16(max m / 63); sc = clamp(rint(s / d), 0, 63), mc = clamp(rint(m /
// dmin), 0, 63) (0 when the divisor is 0); q = clamp(rint((w + dmin*mc) /
// (d*sc)), 0, 15) (0 when d*sc is 0).  Warp per block; lane l holds weights
// 8l .. 8l+7 (sub-block l / 4).
__global__ void __launch_bounds__(256) q4k_quantize_kernel(const float* __restrict__ w, int64_t n_blocks,
                                                           uint8_t* __restrict__ out) {
    __shared__ uint8_t qbuf[8][256];
    __shared__ uint8_t scb[8][8], mcb[8][8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sb = lane >> 2;
    for (int64_t bi = (int64_t)blockIdx.x * 8 + warp; bi < n_blocks; bi += (int64_t)gridDim.x * 8) {
        const float4* src = reinterpret_cast<const float4*>(w + bi * 256 + 8 * lane);
        const float4 a = src[0], b = src[1];
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float mn = v[0], mx = v[0];
#pragma unroll
        for (int i = 1; i < 8; i++) {
            mn = fminf(mn, v[i]);
            mx = fmaxf(mx, v[i]);
        }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        const float m = mn < 0.0f ? -mn : 0.0f;
        const float s = __fdiv_rn(__fadd_rn(mx, m), 15.0f);
        const float maxs = warp_max(s);
        const float maxm = warp_max(m);
        const __half dh = __float2half_rn(__fdiv_rn(maxs, 63.0f));
        const __half mh = __float2half_rn(__fdiv_rn(maxm, 63.0f));
        const float df = __half2float(dh), mf = __half2float(mh);
        const int sc = df > 0.0f ? (int)fminf(fmaxf(rintf(__fdiv_rn(s, df)), 0.0f), 63.0f) : 0;
        const int mc = mf > 0.0f ? (int)fminf(fmaxf(rintf(__fdiv_rn(m, mf)), 0.0f), 63.0f) : 0;
        const float step = __fmul_rn(df, (float)sc);
        const float base = __fmul_rn(mf, (float)mc);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            int q = 0;
            if (step > 0.0f) q = (int)fminf(fmaxf(rintf(__fdiv_rn(__fadd_rn(v[i], base), step)), 0.0f), 15.0f);
            qbuf[warp][8 * lane + i] = (uint8_t)q;
        }
        if ((lane & 3) == 0) {
            scb[warp][sb] = (uint8_t)sc;
            mcb[warp][sb] = (uint8_t)mc;
        }
        __syncwarp();
        // 36 words: d | dmin, three words of scale bytes, 32 words of codes
#pragma unroll
        for (int wi = lane; wi < 36; wi += 32) {
            uint32_t word = 0;
            if (wi == 0) {
                word = (uint32_t)__half_as_ushort(dh) | ((uint32_t)__half_as_ushort(mh) << 16);
            } else if (wi < 4) {
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const int sbyte = 4 * (wi - 1) + c;  // scale byte index 0..11
                    uint32_t byte;
                    if (sbyte < 4)
                        byte = (scb[warp][sbyte] & 63u) | ((uint32_t)(scb[warp][sbyte + 4] >> 4) << 6);
                    else if (sbyte < 8)
                        byte = (mcb[warp][sbyte - 4] & 63u) | ((uint32_t)(mcb[warp][sbyte] >> 4) << 6);
                    else
                        byte = (scb[warp][sbyte - 4] & 15u) | ((uint32_t)(mcb[warp][sbyte - 4] & 15u) << 4);
                    word |= (byte & 0xffu) << (8 * c);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const int qb = 4 * (wi - 4) + c;  // code byte 32c' + l
                    const int cc = qb >> 5, l = qb & 31;
                    const uint32_t byte = (uint32_t)qbuf[warp][64 * cc + l] | ((uint32_t)qbuf[warp][64 * cc + 32 + l] << 4);
                    word |= byte << (8 * c);
                }
            }
            reinterpret_cast<uint32_t*>(out + bi * kQ4Bytes)[wi] = word;
        }
        __syncwarp();
    }
}

cudaError_t launch_q4k_quantize(const float* w, int64_t n_blocks, uint8_t* out, cudaStream_t st) {
    int64_t grid = (n_blocks + 7) / 8;
    if (grid > 152 * 64) grid = 152 * 64;
    q4k_quantize_kernel<<<(unsigned)grid, 256, 0, st>>>(w, n_blocks, out);
    return cudaGetLastError();
}

// ====================================================================== dot products

constexpr int kQ4Threads = 256;

// Staged activation rows.  A row of K activations (nsub = K/32 sub-blocks) is kept as
// float4 groups ordered [w][s]: group w (values 4w..4w+3) of sub-block s is float4 number
// w * nsub + s.  A lane that owns sub-block s reads groups w = 0..7 in order, so at each
// step the lanes of a warp (consecutive s) read consecutive 16-byte groups.
__device__ __forceinline__ int q4_stage_pos(int e, int nsub) {
    const int sb = e >> 5, c = e & 31;
    return (((c >> 2) * nsub + sb) << 2) | (c & 3);
}

// Dot of one 32-weight sub-block j of the 16-byte-aligned block `blk` (global or shared
// memory) with the 32 activations of sub-block s of a staged row a4 (nsub sub-blocks,
// shared memory) whose sum is asum.
__device__ __forceinline__ float q4k_sub_dot(const uint8_t* blk, int j, const float4* a4, int nsub, int s,
                                             float asum) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
    const float dm = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
    const int jj = j & 3;
    const uint32_t sy = (hdr.y >> (8 * jj)) & 0xffu, sz = (hdr.z >> (8 * jj)) & 0xffu, sw = (hdr.w >> (8 * jj)) & 0xffu;
    const uint32_t sc = j < 4 ? (sy & 63u) : ((sw & 15u) | ((sy >> 6) << 4));
    const uint32_t mn = j < 4 ? (sz & 63u) : ((sw >> 4) | ((sz >> 6) << 4));
    const uint4* qs = reinterpret_cast<const uint4*>(blk + 16 + 32 * (j >> 1));
    const int sh = 4 * (j & 1);
    const uint4 q0 = qs[0], q1 = qs[1];
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; w++) {
        const float4 x = a4[w * nsub + s];
        const uint32_t v = qw[w] >> sh;
        acc = fmaf((float)(v & 15u), x.x, acc);
        acc = fmaf((float)((v >> 8) & 15u), x.y, acc);
        acc = fmaf((float)((v >> 16) & 15u), x.z, acc);
        acc = fmaf((float)((v >> 24) & 15u), x.w, acc);
    }
    return d * (float)sc * acc - dm * (float)mn * asum;
}

// Stage n activations (rows of K, K a multiple of 256) as fp32 in the [w][s] order above,
// and the sum of each 32-value sub-block, added in element order (block-wide).  Each
// thread issues up to eight loads before it stores any of them.
template <class Load>
__device__ __forceinline__ void stage_row(Load ld, int n, int K, float* a, float* asum) {
    const int nsub = K >> 5;
#pragma unroll 1
    for (int i0 = threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int i = i0 + u * blockDim.x;
            v[u] = i < n ? ld(i) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int i = i0 + u * blockDim.x;
            if (i < n) {
                const int r = i / K, e = i - r * K;
                a[(size_t)r * K + q4_stage_pos(e, nsub)] = v[u];
            }
        }
    }
    __syncthreads();
    for (int g = threadIdx.x; g < n / 32; g += blockDim.x) {
        const int r = g / nsub, sb = g - r * nsub;
        const float* row = a + (size_t)r * K;
        float s = 0.0f;
#pragma unroll 8
        for (int i = 0; i < 32; i++) s += row[q4_stage_pos(32 * sb + i, nsub)];
        asum[g] = s;
    }
    __syncthreads();
}

__device__ __forceinline__ float load_x_f32(const void* x, int x_dtype, size_t i) {
    if (x_dtype == QS_BF16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(x)[i] << 16);
    return reinterpret_cast<const float*>(x)[i];
}

// Dot of a row of nb blocks with the staged activations: lanes stride over the row's
// 8*nb sub-blocks; one fixed butterfly sum over the warp.  Every lane gets the result.
__device__ __forceinline__ float q4k_row_dot(const uint8_t* row, int nb, const float* a, const float* asum) {
    const int lane = threadIdx.x & 31;
    const float4* a4 = reinterpret_cast<const float4*>(a);
    const int nsub = 8 * nb;
    float acc = 0.0f;
    for (int s = lane; s < nsub; s += 32)
        acc += q4k_sub_dot(row + (size_t)(s >> 3) * kQ4Bytes, s & 7, a4, nsub, s, asum[s]);
    return warp_sum(acc);
}

// ====================================================================== gate/up + SwiGLU

struct alignas(16) Q4GateUpSmem {
    uint64_t bar;
    int32_t expert;
    int32_t ok;
    int32_t wcnt[kQ4Threads / 32];
};

// grid.x = max_active * (F / R); block kQ4Threads.
// dynamic smem: Q4GateUpSmem | x f32[H] | x sums f32[H/32] | gate and up tiles 2 * R * rowbytes.
__global__ void __launch_bounds__(kQ4Threads) q4k_gateup_kernel(const void* __restrict__ x, int x_dtype, int H, int E,
                                                                 int k, int F, int R, const uint8_t* __restrict__ experts,
                                                                 int64_t stride, const int32_t* __restrict__ offsets,
                                                                 const int32_t* __restrict__ perm, float* h_out) {
    extern __shared__ __align__(128) uint8_t smem[];
    Q4GateUpSmem& S = *reinterpret_cast<Q4GateUpSmem*>(smem);
    float* xa = reinterpret_cast<float*>(smem + sizeof(Q4GateUpSmem));
    float* xsum = xa + H;
    uint8_t* wbuf = reinterpret_cast<uint8_t*>(xsum + H / 32);
    const int nb = H / kBlockWeights;
    const int rowbytes = nb * kQ4Bytes;
    const int tiles = F / R;
    const int a = blockIdx.x / tiles, tile = blockIdx.x % tiles;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // the a-th active expert (ascending id): block-wide exclusive count of active experts
    if (threadIdx.x == 0) S.expert = -1;
    __syncthreads();
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const bool act = e < E && offsets[e + 1] > offsets[e];
        const unsigned bal = __ballot_sync(0xffffffffu, act);
        if (lane == 0) S.wcnt[warp] = __popc(bal);
        __syncthreads();
        int before = base, tot = 0;
        for (int w = 0; w < kQ4Threads / 32; w++) {
            if (w < warp) before += S.wcnt[w];
            tot += S.wcnt[w];
        }
        before += __popc(bal & ((1u << lane) - 1u));
        if (act && before == a) S.expert = e;
        base += tot;
        __syncthreads();
    }
    const int e = S.expert;
    if (e < 0) return;  // fewer active experts than the grid allows for

    const uint8_t* gate_rows = experts + (int64_t)e * stride + (int64_t)tile * R * rowbytes;
    const uint8_t* up_rows = gate_rows + (int64_t)F * rowbytes;
    const uint32_t tile_bytes = (uint32_t)R * rowbytes;
    if (threadIdx.x == 0) {
        mbar_init(&S.bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&S.bar, 2 * tile_bytes);
        bulk_g2s(wbuf, gate_rows, tile_bytes, &S.bar);
        bulk_g2s(wbuf + tile_bytes, up_rows, tile_bytes, &S.bar);
    }
    bool waited = false;
    const int j0 = offsets[e], j1 = offsets[e + 1];
    for (int j = j0; j < j1; j++) {
        const int entry = perm[j];
        const int t = entry / k;
        stage_row([&](int i) { return load_x_f32(x, x_dtype, (size_t)t * H + i); }, H, H, xa, xsum);
        if (!waited) {
            if (threadIdx.x == 0) S.ok = mbar_wait(&S.bar, 0) ? 1 : 0;
            __syncthreads();
            if (!S.ok) return;  // the copy never completed: outputs left unwritten
            // every thread observes the completed phase (its first poll succeeds), which makes
            // the copied bytes visible to it
            (void)mbar_wait(&S.bar, 0);
            waited = true;
        }
        for (int r = warp; r < R; r += kQ4Threads / 32) {
            const float g = q4k_row_dot(wbuf + (size_t)r * rowbytes, nb, xa, xsum);
            const float u = q4k_row_dot(wbuf + tile_bytes + (size_t)r * rowbytes, nb, xa, xsum);
            if (lane == 0) h_out[(size_t)entry * F + tile * R + r] = silu(g) * u;
        }
        __syncthreads();  // xa is rewritten for the next token
    }
    if (!waited) {  // never leave a copy in flight into freed shared memory
        if (threadIdx.x == 0) (void)mbar_wait(&S.bar, 0);
        __syncthreads();
    }
}

// ====================================================================== down + routing-weight combine

constexpr int kQ4DownRowsMax = 16;

// grid (H / rows, T); block kQ4Threads; rows is 4 or 16 (a divisor of H).  dynamic smem:
// h f32[k][F] | h sums f32[k][F/32] | slot expert i32[k] | slot weight f32[k].  A warp
// takes (row, slot) pairs and leaves each dot in shared memory; then one thread per row
// forms out[t, r] = sum over slots (in slot order) of p * (Wd_e h) -- stored, not added.
__global__ void __launch_bounds__(kQ4Threads) q4k_down_kernel(int H, int k, int F, int rows,
                                                              const uint8_t* __restrict__ experts,
                                                              int64_t stride, const float* __restrict__ h,
                                                              const int32_t* __restrict__ ids,
                                                              const float* __restrict__ pw, float* __restrict__ out) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float dots[kQ4DownRowsMax * 32];  // [row][slot], k <= 32
    float* ha = reinterpret_cast<float*>(smem);
    float* hsum = ha + (size_t)k * F;
    int32_t* se = reinterpret_cast<int32_t*>(hsum + (size_t)k * (F / 32));
    float* sp = reinterpret_cast<float*>(se + k);
    const int t = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nbh = H / kBlockWeights, nbf = F / kBlockWeights;
    const int64_t rb_h = (int64_t)nbh * kQ4Bytes, rb_f = (int64_t)nbf * kQ4Bytes;
    if (threadIdx.x < k) {
        se[threadIdx.x] = ids[(size_t)t * k + threadIdx.x];
        sp[threadIdx.x] = pw[(size_t)t * k + threadIdx.x];
    }
    const float* ht = h + (size_t)t * k * F;
    stage_row([&](int i) { return ht[i]; }, k * F, F, ha, hsum);
#pragma unroll 1
    for (int q = warp; q < rows * k; q += kQ4Threads / 32) {
        const int rr = q / k, j = q - rr * k;
        const int r = blockIdx.x * rows + rr;
        const uint8_t* row = experts + (int64_t)se[j] * stride + 2ll * F * rb_h + (int64_t)r * rb_f;
        const float v = q4k_row_dot(row, nbf, ha + (size_t)j * F, hsum + (size_t)j * (F / 32));
        if (lane == 0) dots[rr * 32 + j] = v;
    }
    __syncthreads();
    if (threadIdx.x < rows) {
        float acc = 0.0f;
        for (int j = 0; j < k; j++) acc = fmaf(sp[j], dots[threadIdx.x * 32 + j], acc);
        out[(size_t)t * H + blockIdx.x * rows + threadIdx.x] = acc;
    }
}

// ====================================================================== launchers

// Opt a kernel in to `bytes` of dynamic shared memory when its dynamic plus static shared
// memory passes the 48 KB a launch gets without the attribute.
static cudaError_t q4_set_smem(const void* fn, size_t bytes) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    if (bytes + fa.sharedSizeBytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

size_t q4k_down_smem(int k, int F) { return (size_t)k * F * 4 + (size_t)k * (F / 32) * 4 + (size_t)k * 8; }

cudaError_t launch_q4k_gateup(const qs_moe_shape& s, const void* x, const uint8_t* experts, int64_t stride,
                              const int32_t* offsets, const int32_t* perm, int T, float* h, cudaStream_t st) {
    const int H = s.hidden, F = s.expert_ffn;
    const int rowbytes = H / kBlockWeights * kQ4Bytes;
    int R = 16;  // rows per tile: both staged tiles together <= ~72 KB
    while (R > 1 && (size_t)2 * R * rowbytes > 72 * 1024) R >>= 1;
    const size_t smem = sizeof(Q4GateUpSmem) + (size_t)H * 4 + (size_t)(H / 32) * 4 + 2 * (size_t)R * rowbytes;
    cudaError_t err = q4_set_smem((const void*)q4k_gateup_kernel, smem);
    if (err != cudaSuccess) return err;
    const int max_active = std::min(s.n_experts, T * s.top_k);
    q4k_gateup_kernel<<<max_active * (F / R), kQ4Threads, smem, st>>>(x, s.x_dtype, H, s.n_experts, s.top_k, F, R,
                                                                       experts, stride, offsets, perm, h);
    return cudaGetLastError();
}

cudaError_t launch_q4k_down(const qs_moe_shape& s, const uint8_t* experts, int64_t stride, const float* h,
                            const int32_t* ids, const float* pw, int T, float* out, cudaStream_t st) {
    const size_t smem = q4k_down_smem(s.top_k, s.expert_ffn);
    cudaError_t err = q4_set_smem((const void*)q4k_down_kernel, smem);
    if (err != cudaSuccess) return err;
    // few tokens: 4 output rows per CTA, so that the grid covers the SMs; many tokens: 16, so
    // that the h rows each CTA stages are shared by more output rows
    const int rows = T <= 16 ? 4 : kQ4DownRowsMax;
    dim3 grid(s.hidden / rows, T);
    q4k_down_kernel<<<grid, kQ4Threads, smem, st>>>(s.hidden, s.top_k, s.expert_ffn, rows, experts, stride, h, ids,
                                                    pw, out);
    return cudaGetLastError();
}

}  // namespace qs

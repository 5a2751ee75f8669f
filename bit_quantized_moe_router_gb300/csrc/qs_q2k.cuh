// qs_q2k.cuh -- Q2_K dot-product and routing device functions shared by the
// per-step kernels and the persistent decode kernel.
#pragma once

#include "qs_common.cuh"

namespace qs {

// One warp: top-k of E <= 1024 logits (k <= E), descending, ties to the lower
// index; softmax over the selected logits.  Every returned id is in [0, E).
__device__ __forceinline__ void topk_softmax_warp(const float* l, int E, int k, int32_t* ids_out, float* w_out) {
    const int lane = threadIdx.x & 31;
    float v[32];
#pragma unroll
    for (int m = 0; m < 32; m++) {
        const int e = lane + 32 * m;
        const float lv = (e < E) ? __ldcg(l + e) : -INFINITY;
        v[m] = (lv == lv) ? lv : -INFINITY;  // a NaN logit ranks last, so every chosen id is in range
    }
    uint32_t taken = 0;
    float my_l = -INFINITY;
    int my_id = 0;
    for (int j = 0; j < k; j++) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int m = 0; m < 32; m++) {
            const int e = lane + 32 * m;
            if (e < E && !((taken >> m) & 1u) && (v[m] > bv || (v[m] == bv && e < bi))) {
                bv = v[m];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi != 0x7fffffff && (bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            my_l = bv;
            my_id = bi;
        }
    }
    const float lmax = __shfl_sync(0xffffffffu, my_l, 0);
    const float ex = (lane < k) ? expf(my_l - lmax) : 0.0f;
    const float den = warp_sum(ex);
    if (lane < k) {
        ids_out[lane] = my_id;
        w_out[lane] = ex / den;
    }
}

// ====================================================================== Q2_K chunk dot

// A thread's slice of one token's int16 activations: chunk u of block b.
struct XFrag {
    int32_t v[4][4][2];  // [shift j][word w][pair]: (x[p], x[p+1]) and (x[p+2], x[p+3])
    int32_t xs[4];       // sum of the 16 activations of sub-block j
};

// xq: the token's int16 activations in shared memory (8-byte aligned).
__device__ __forceinline__ void load_xfrag(const int16_t* xq, int b, int u, XFrag& f) {
    const int base = 256 * b + 128 * (u >> 1) + 16 * (u & 1);
#pragma unroll
    for (int j = 0; j < 4; j++) {
        int s = 0;
#pragma unroll
        for (int w = 0; w < 4; w++) {
            const uint2 pr = *reinterpret_cast<const uint2*>(xq + base + 32 * j + 4 * w);
            f.v[j][w][0] = (int32_t)pr.x;
            f.v[j][w][1] = (int32_t)pr.y;
            s = dp2a_lo((int32_t)pr.x, 0x0101u, s);
            s = dp2a_lo((int32_t)pr.y, 0x0101u, s);
        }
        f.xs[j] = s;
    }
}

// Fragment layout of int16 activations: chunk c = 4b + u of a row (the 64
// activations chunk u of block b multiplies) is 36 consecutive 32-bit words,
// 144 bytes: words 8j + 2w and 8j + 2w + 1 hold the int16 pairs (x[p], x[p+1])
// and (x[p+2], x[p+3]) with p = 256b + 128(u>>1) + 32j + 16(u&1) + 4w, and word
// 32 + j holds the sum of the 16 activations of shift group j.  A lane reads
// its fragment with nine 16-byte loads; lanes reading consecutive chunks hit
// distinct banks.
constexpr int kFragWords = 36;

__device__ __forceinline__ void load_xfrag_f(const uint32_t* frag, XFrag& f) {
    const uint4* q = reinterpret_cast<const uint4*>(frag);
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const uint4 a = q[2 * j], b = q[2 * j + 1];
        f.v[j][0][0] = (int32_t)a.x;
        f.v[j][0][1] = (int32_t)a.y;
        f.v[j][1][0] = (int32_t)a.z;
        f.v[j][1][1] = (int32_t)a.w;
        f.v[j][2][0] = (int32_t)b.x;
        f.v[j][2][1] = (int32_t)b.y;
        f.v[j][3][0] = (int32_t)b.z;
        f.v[j][3][1] = (int32_t)b.w;
    }
    const uint4 s = q[8];
    f.xs[0] = (int32_t)s.x;
    f.xs[1] = (int32_t)s.y;
    f.xs[2] = (int32_t)s.z;
    f.xs[3] = (int32_t)s.w;
}

// Word index (within a row's fragment array) and half of activation position p.
__device__ __forceinline__ void frag_pos(int p, int& word, int& half) {
    const int b = p >> 8, h = (p >> 7) & 1, j = (p >> 5) & 3, u1 = (p >> 4) & 1, w = (p >> 2) & 3, e = p & 3;
    word = (4 * b + 2 * h + u1) * kFragWords + 8 * j + 2 * w + (e >> 1);
    half = e & 1;
}

// The words of one Q2_K block that chunk u reads: its 16 quant bytes, the 8 scale bytes of
// its half, and d | dmin.
struct Q2Chunk {
    uint32_t q[4];
    uint32_t sca, scb, dd;
};

// Chunk u of the block at blk (4-byte aligned; shared or global memory).
__device__ __forceinline__ void load_q2chunk(const uint8_t* blk, int u, Q2Chunk& c) {
    const uint32_t* b32 = reinterpret_cast<const uint32_t*>(blk);
#pragma unroll
    for (int w = 0; w < 4; w++) c.q[w] = b32[4 + 4 * u + w];
    c.sca = b32[2 * (u >> 1)];
    c.scb = b32[2 * (u >> 1) + 1];
    c.dd = b32[20];
}

// The same words from global memory through the read-only path.
__device__ __forceinline__ void load_q2chunk_global(const uint8_t* blk, int u, Q2Chunk& c) {
    const uint32_t* b32 = reinterpret_cast<const uint32_t*>(blk);
#pragma unroll
    for (int w = 0; w < 4; w++) c.q[w] = __ldg(b32 + 4 + 4 * u + w);
    c.sca = __ldg(b32 + 2 * (u >> 1));
    c.scb = __ldg(b32 + 2 * (u >> 1) + 1);
    c.dd = __ldg(b32 + 20);
}

// Partial dot of chunk u of a block (its words in c) with the thread's activations:
// d * sum sc_lo*S - dmin * sum sc_hi*X (unscaled by s_x).
// Integer sums are exact, so the four words' partial sums are formed independently (short
// dependency chains for the scheduler) and added afterwards; the result is the same bits.
__device__ __forceinline__ float q2k_chunk_dot(const Q2Chunk& c, int u, const XFrag& f) {
    const int sh0 = 8 * (u & 1);
    int plo = 0, phi = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const uint32_t mask = 0x03030303u << (2 * j);
        int tw[4];
#pragma unroll
        for (int w = 0; w < 4; w++) {
            const uint32_t v = c.q[w] & mask;
            tw[w] = dp2a_hi(f.v[j][w][1], v, dp2a_lo(f.v[j][w][0], v, 0));
        }
        int t = (tw[0] + tw[1]) + (tw[2] + tw[3]);
        t >>= 2 * j;
        const uint32_t sc = ((j < 2 ? c.sca : c.scb) >> (sh0 + 16 * (j & 1))) & 0xffu;
        plo += (int)(sc & 15u) * t;
        phi += (int)(sc >> 4) * f.xs[j];
    }
    const float d = __half2float(__ushort_as_half((unsigned short)(c.dd & 0xffffu)));
    const float dm = __half2float(__ushort_as_half((unsigned short)(c.dd >> 16)));
    return __fmaf_rn(d, (float)plo, __fmul_rn(-dm, (float)phi));
}

// Partial dots of chunk u of two blocks (a, b: e.g. a gate row's and an up row's) with the
// activations of one fragment in shared memory (kFragWords layout), read one shift group at a
// time so that few registers are live.  Each result is the same bits as q2k_chunk_dot's.
__device__ __forceinline__ void q2k_chunk_dot2_f(const Q2Chunk& a, const Q2Chunk& b, int u, const uint32_t* frag,
                                                 float& da, float& db) {
    const uint4* q = reinterpret_cast<const uint4*>(frag);
    const uint4 xs = q[8];
    const int xsj[4] = {(int)xs.x, (int)xs.y, (int)xs.z, (int)xs.w};
    const int sh0 = 8 * (u & 1);
    int alo = 0, ahi = 0, blo = 0, bhi = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const uint4 p0 = q[2 * j], p1 = q[2 * j + 1];
        const int32_t x[4][2] = {{(int32_t)p0.x, (int32_t)p0.y}, {(int32_t)p0.z, (int32_t)p0.w},
                                 {(int32_t)p1.x, (int32_t)p1.y}, {(int32_t)p1.z, (int32_t)p1.w}};
        const uint32_t mask = 0x03030303u << (2 * j);
        int ta[4], tb[4];
#pragma unroll
        for (int w = 0; w < 4; w++) {
            const uint32_t va = a.q[w] & mask, vb = b.q[w] & mask;
            ta[w] = dp2a_hi(x[w][1], va, dp2a_lo(x[w][0], va, 0));
            tb[w] = dp2a_hi(x[w][1], vb, dp2a_lo(x[w][0], vb, 0));
        }
        const int sa = ((ta[0] + ta[1]) + (ta[2] + ta[3])) >> (2 * j);
        const int sb = ((tb[0] + tb[1]) + (tb[2] + tb[3])) >> (2 * j);
        const uint32_t sca = ((j < 2 ? a.sca : a.scb) >> (sh0 + 16 * (j & 1))) & 0xffu;
        const uint32_t scb = ((j < 2 ? b.sca : b.scb) >> (sh0 + 16 * (j & 1))) & 0xffu;
        alo += (int)(sca & 15u) * sa;
        ahi += (int)(sca >> 4) * xsj[j];
        blo += (int)(scb & 15u) * sb;
        bhi += (int)(scb >> 4) * xsj[j];
    }
    const float d_a = __half2float(__ushort_as_half((unsigned short)(a.dd & 0xffffu)));
    const float m_a = __half2float(__ushort_as_half((unsigned short)(a.dd >> 16)));
    const float d_b = __half2float(__ushort_as_half((unsigned short)(b.dd & 0xffffu)));
    const float m_b = __half2float(__ushort_as_half((unsigned short)(b.dd >> 16)));
    da = __fmaf_rn(d_a, (float)alo, __fmul_rn(-m_a, (float)ahi));
    db = __fmaf_rn(d_b, (float)blo, __fmul_rn(-m_b, (float)bhi));
}

// Partial dot of chunk u of the block at blk (shared memory, 4-byte aligned).
__device__ __forceinline__ float q2k_chunk_dot(const uint8_t* blk, int u, const XFrag& f) {
    Q2Chunk c;
    load_q2chunk(blk, u, c);
    return q2k_chunk_dot(c, u, f);
}


}  // namespace qs

// qs_fmt.cuh -- the routed-weight formats of the persistent decode kernel: per 64-weight chunk
// of a super-block, the words a lane loads, the int16 activation fragment it multiplies, and
// the dot product.  Integer sums are exact; d and dmin are applied once per chunk in fp32.
//
// Q2_K (84 bytes per 256 weights): the chunk dot and fragment layout of qs_q2k.cuh.
// Q4_K (144 bytes per 256 weights, GGUF layout, 16-byte aligned blocks):
//   d (fp16) | dmin (fp16) | scales[12] | qs[128]; eight 32-weight sub-blocks j with 6-bit
//   scale and min: j < 4: sc = S[j] & 63, m = S[j + 4] & 63; j >= 4: sc = (S[j + 4] & 15) |
//   (S[j - 4] >> 6) << 4, m = (S[j + 4] >> 4) | (S[j] >> 6) << 4; weight 64c + l is the low
//   nibble of qs[32c + l] (sub-block 2c), weight 64c + 32 + l its high nibble (sub-block
//   2c + 1); w = d * sc * q - dmin * m.  Chunk c is sub-blocks 2c and 2c + 1: one 16-byte load
//   of the block head and two of the chunk's 32 code bytes.  Its fragment is the 64 int16
//   activations in order (32 words) and the two 32-value sums (words 32, 33).
#pragma once

#include "qs_q2k.cuh"

namespace qs {

enum WeightFmt { kFmtQ2K = 0, kFmtQ4K = 1 };

template <int FMT>
struct FmtOps;

template <>
struct FmtOps<kFmtQ2K> {
    static constexpr int kBlock = kBlockBytes;
    using Chunk = Q2Chunk;
    using Frag = XFrag;
    __device__ static __forceinline__ void load(const uint8_t* blk, int u, Chunk& c) { load_q2chunk_global(blk, u, c); }
    __device__ static __forceinline__ void load_frag(const uint32_t* f, Frag& x) { load_xfrag_f(f, x); }
    __device__ static __forceinline__ float dot(const Chunk& c, int u, const Frag& f) { return q2k_chunk_dot(c, u, f); }
    __device__ static __forceinline__ void dot2(const Chunk& a, const Chunk& b, int u, const uint32_t* f, float& da,
                                                float& db) {
        q2k_chunk_dot2_f(a, b, u, f, da, db);
    }
    // This lane's 8 int16 activations wq at position p (p % 8 == 0) of a row's fragments, sum =
    // their sum.  Lanes hold consecutive 8-value groups; every lane of the warp calls it.
    __device__ static __forceinline__ void put8(uint32_t* row, int p, const uint32_t (&wq)[4], int sum, bool live) {
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        if (live) {
            int word, half;
            frag_pos(p, word, half);
            *reinterpret_cast<uint4*>(row + word) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
            if ((p & 15) == 0) row[(word / kFragWords) * kFragWords + 32 + ((p >> 5) & 3)] = (uint32_t)sum;
        }
    }
};

struct Q4Chunk {
    uint32_t q[8];   // the chunk's 32 code bytes
    uint32_t s[3];   // scales[12]
    uint32_t dd;     // d | dmin << 16
};
struct Q4Frag {
    int32_t v[32];   // int16 pairs of the 64 activations, in order
    int32_t xs[2];   // sums of activations 0..31 and 32..63
};

// Scale and min of sub-block j from the 12 scale bytes.
__device__ __forceinline__ void q4k_scale_min(const uint32_t (&s)[3], int j, int& sc, int& m) {
    auto S = [&](int i) -> int {  // byte i (selects, not an indexed array: no local memory)
        const uint32_t w = i < 4 ? s[0] : (i < 8 ? s[1] : s[2]);
        return (int)((w >> (8 * (i & 3))) & 0xffu);
    };
    if (j < 4) {
        sc = S(j) & 63;
        m = S(j + 4) & 63;
    } else {
        sc = (S(j + 4) & 15) | ((S(j - 4) >> 6) << 4);
        m = (S(j + 4) >> 4) | ((S(j) >> 6) << 4);
    }
}

// Dot of chunk u's 64 weights with activations given as 32 pair words v and two sums.
template <class V>
__device__ __forceinline__ float q4k_chunk_dot_v(const Q4Chunk& c, int u, V v, int xs0, int xs1) {
    int tl[8], th[8];
#pragma unroll
    for (int w = 0; w < 8; w++) {
        const uint32_t lo = c.q[w] & 0x0f0f0f0fu, hi = (c.q[w] >> 4) & 0x0f0f0f0fu;
        tl[w] = dp2a_hi(v(2 * w + 1), lo, dp2a_lo(v(2 * w), lo, 0));
        th[w] = dp2a_hi(v(16 + 2 * w + 1), hi, dp2a_lo(v(16 + 2 * w), hi, 0));
    }
    const int slo = ((tl[0] + tl[1]) + (tl[2] + tl[3])) + ((tl[4] + tl[5]) + (tl[6] + tl[7]));
    const int shi = ((th[0] + th[1]) + (th[2] + th[3])) + ((th[4] + th[5]) + (th[6] + th[7]));
    int sc0, m0, sc1, m1;
    q4k_scale_min(c.s, 2 * u, sc0, m0);
    q4k_scale_min(c.s, 2 * u + 1, sc1, m1);
    const int plo = sc0 * slo + sc1 * shi;  // |.| < 2 * 63 * 32 * 15 * 32767 < 2^31
    const int phi = m0 * xs0 + m1 * xs1;
    const float d = __half2float(__ushort_as_half((unsigned short)(c.dd & 0xffffu)));
    const float dm = __half2float(__ushort_as_half((unsigned short)(c.dd >> 16)));
    return __fmaf_rn(d, (float)plo, __fmul_rn(-dm, (float)phi));
}

template <>
struct FmtOps<kFmtQ4K> {
    static constexpr int kBlock = 144;
    using Chunk = Q4Chunk;
    using Frag = Q4Frag;
    __device__ static __forceinline__ void load(const uint8_t* blk, int u, Chunk& c) {
        const uint4* b = reinterpret_cast<const uint4*>(blk);
        const uint4 h = __ldg(b), a0 = __ldg(b + 1 + 2 * u), a1 = __ldg(b + 2 + 2 * u);
        c.dd = h.x;
        c.s[0] = h.y;
        c.s[1] = h.z;
        c.s[2] = h.w;
        c.q[0] = a0.x; c.q[1] = a0.y; c.q[2] = a0.z; c.q[3] = a0.w;
        c.q[4] = a1.x; c.q[5] = a1.y; c.q[6] = a1.z; c.q[7] = a1.w;
    }
    __device__ static __forceinline__ void load_frag(const uint32_t* f, Frag& x) {
        const uint4* q = reinterpret_cast<const uint4*>(f);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint4 a = q[i];
            x.v[4 * i] = (int32_t)a.x;
            x.v[4 * i + 1] = (int32_t)a.y;
            x.v[4 * i + 2] = (int32_t)a.z;
            x.v[4 * i + 3] = (int32_t)a.w;
        }
        const uint2 s = reinterpret_cast<const uint2*>(f)[16];
        x.xs[0] = (int32_t)s.x;
        x.xs[1] = (int32_t)s.y;
    }
    __device__ static __forceinline__ float dot(const Chunk& c, int u, const Frag& f) {
        return q4k_chunk_dot_v(c, u, [&](int i) { return f.v[i]; }, f.xs[0], f.xs[1]);
    }
    // Two chunks against one fragment in shared memory, its words read where they are used
    // (few live registers).
    __device__ static __forceinline__ void dot2(const Chunk& a, const Chunk& b, int u, const uint32_t* fp, float& da,
                                                float& db) {
        const int32_t* f = reinterpret_cast<const int32_t*>(fp);
        const int2 xs = reinterpret_cast<const int2*>(fp)[16];
        da = q4k_chunk_dot_v(a, u, [&](int i) { return f[i]; }, xs.x, xs.y);
        db = q4k_chunk_dot_v(b, u, [&](int i) { return f[i]; }, xs.x, xs.y);
    }
    __device__ static __forceinline__ void put8(uint32_t* row, int p, const uint32_t (&wq)[4], int sum, bool live) {
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (live) {
            uint32_t* ch = row + (p >> 6) * kFragWords;
            *reinterpret_cast<uint4*>(ch + ((p & 63) >> 1)) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
            if ((p & 31) == 0) ch[32 + ((p >> 5) & 1)] = (uint32_t)sum;
        }
    }
};

}  // namespace qs

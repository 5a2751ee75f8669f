/*
 * qs_oracle.c -- plain, slow CPU oracle of the Q2_K mixture-of-experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links or calls this
 * file; only the tests, the smoke check and the bench's CPU-baseline leg do.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * Everything is computed in double precision, in the plain order of the
 * definition: decode each weight from its block, dot with the widened input,
 * route, SwiGLU, weighted sum, gated shared expert.  The one exception is the
 * Q2_K *encoder* (qso_q2k_quantize_rows), whose integer decisions are taken in
 * fp32 with a fixed operation order so that a device encoder taking the same
 * decisions in fp32 can be compared bit for bit.
 *
 * Sources of the definition:
 *  - QuarkStar (q36) README, "Model Weights" and DwarfStar (ds4) page, "Model
 *    Weights": only routed experts are 2-bit; shared experts, projections and
 *    routing stay in higher precision; down (and here gate/up) is Q2_K.
 *  - QuarkStar (q36) README, "Acknowledgements": GGUF quant layouts are kept,
 *    which fixes the reading of the Q2_K byte order below.
 *  - Quasar (q27) README, "Architecture facts": the FFN is SwiGLU.
 *  - The workload statement of the layer: top-k experts by a router GEMV and
 *    softmax, routing weights summing to 1, Q2_K blocks of 256 weights in 84
 *    bytes (scales[16], qs[64], fp16 d, fp16 dmin), dequantisation
 *    w = d*(sc&15)*q - dmin*(sc>>4), weighted sum plus a sigmoid-gated bf16
 *    shared expert.
 *
 * Readings taken where the sources are silent:
 *  - byte order of a block: scales[0..15] | qs[16..79] | d (fp16 LE, bytes
 *    80-81) | dmin (fp16 LE, bytes 82-83);
 *  - weight i = 128*h + 32*j + l (h in 0..1, j in 0..3, l in 0..31) is bits
 *    2j..2j+1 of qs[32*h + l] and uses scales[i/16]; low nibble = scale,
 *    high nibble = min;
 *  - routing: top-k of the logits, ties to the lower expert index, ids in
 *    descending-logit order, weights = softmax over the k selected logits;
 *  - shared expert gate: scalar sigmoid(w_sg . x) per token.
 *
 * Pins (tests that tie this file to something other than itself): hand-built
 * blocks with closed-form values, single-bit probes of the packing order, a
 * pack/unpack round trip, textbook special cases of the layer (one expert =
 * a SwiGLU MLP, diagonal experts = elementwise SwiGLU, zero router = uniform
 * weights, zero gate vector = gate 1/2), brute-force top-k and grouping.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QSO_BLOCK_BYTES 84
#define QSO_BLOCK_WEIGHTS 256

/* ------------------------------------------------------------------ */
/* storage types                                                        */
/* ------------------------------------------------------------------ */

/* IEEE binary16 bit pattern -> double (exact). */
double qso_half_to_double(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    }
    return s ? -v : v;
}

/* bfloat16 bit pattern -> double (exact: the upper half of an fp32). */
double qso_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* fp32 -> IEEE binary16, round to nearest, ties to even (from the IEEE 754
 * definition: scale to an integer significand and round once). */
uint16_t qso_float_to_half(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);  /* NaN */
    double a = fabs((double)f);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);                      /* rounds past 65504 */
    if (a < ldexp(1.0, -14)) {                                                /* subnormal range */
        double m = nearbyint(ldexp(a, 24));                                   /* may reach 1024 = min normal */
        return (uint16_t)(sign | (uint16_t)m);
    }
    int ex;
    frexp(a, &ex);                                                            /* a = fr * 2^ex, fr in [0.5,1) */
    int E = ex - 1;                                                           /* a = 1.f * 2^E */
    double m = nearbyint((ldexp(a, -E) - 1.0) * 1024.0);
    if (m >= 1024.0) { m = 0.0; E += 1; }
    if (E + 15 >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)m);
}

/* ------------------------------------------------------------------ */
/* Q2_K block                                                           */
/* ------------------------------------------------------------------ */

/* Split one 84-byte block into its fields: 16 scale bytes, 256 codes in
 * 0..3 (in weight order), and the fp16 bit patterns of d and dmin. */
void qso_q2k_unpack(const uint8_t *blk, uint8_t *scales, uint8_t *q, uint16_t *d, uint16_t *dmin) {
    for (int s = 0; s < 16; s++) scales[s] = blk[s];
    for (int i = 0; i < QSO_BLOCK_WEIGHTS; i++) {
        int h = i / 128, j = (i % 128) / 32, l = i % 32;
        q[i] = (uint8_t)((blk[16 + 32 * h + l] >> (2 * j)) & 3);
    }
    *d = (uint16_t)(blk[80] | (blk[81] << 8));
    *dmin = (uint16_t)(blk[82] | (blk[83] << 8));
}

/* Inverse of qso_q2k_unpack. */
void qso_q2k_pack(const uint8_t *scales, const uint8_t *q, uint16_t d, uint16_t dmin, uint8_t *blk) {
    memset(blk, 0, QSO_BLOCK_BYTES);
    for (int s = 0; s < 16; s++) blk[s] = scales[s];
    for (int i = 0; i < QSO_BLOCK_WEIGHTS; i++) {
        int h = i / 128, j = (i % 128) / 32, l = i % 32;
        blk[16 + 32 * h + l] |= (uint8_t)((q[i] & 3) << (2 * j));
    }
    blk[80] = (uint8_t)(d & 0xff);
    blk[81] = (uint8_t)(d >> 8);
    blk[82] = (uint8_t)(dmin & 0xff);
    blk[83] = (uint8_t)(dmin >> 8);
}

/* Decode one row of K weights (K/256 consecutive blocks) to double:
 * w = d*(sc & 15)*q - dmin*(sc >> 4), exact in double. */
void qso_q2k_dequant_row(const uint8_t *row, int64_t K, double *w) {
    uint8_t sc[16], q[256];
    uint16_t dh, mh;
    for (int64_t b = 0; b < K / QSO_BLOCK_WEIGHTS; b++) {
        qso_q2k_unpack(row + b * QSO_BLOCK_BYTES, sc, q, &dh, &mh);
        double d = qso_half_to_double(dh), dmin = qso_half_to_double(mh);
        for (int i = 0; i < QSO_BLOCK_WEIGHTS; i++) {
            int s = i / 16;
            w[b * QSO_BLOCK_WEIGHTS + i] = d * (double)(sc[s] & 15) * (double)q[i] - dmin * (double)(sc[s] >> 4);
        }
    }
}

void qso_q2k_dequant_rows(const uint8_t *rows, int64_t n_rows, int64_t K, double *w) {
    int64_t row_bytes = K / QSO_BLOCK_WEIGHTS * QSO_BLOCK_BYTES;
    for (int64_t r = 0; r < n_rows; r++) qso_q2k_dequant_row(rows + r * row_bytes, K, w + r * K);
}

static float clampf_(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* Round-to-nearest Q2_K encoder (set-up step, not part of the layer).
 * Per 16-weight sub-block: m = max(0, -min w), s = (max w + m)/3.
 * Per block: d = fp16(max s / 15), dmin = fp16(max m / 15);
 * sc_lo = clamp(rint(s/d),0,15), sc_hi = clamp(rint(m/dmin),0,15) (0 when the
 * divisor is 0); q = clamp(rint((w + dmin*sc_hi)/(d*sc_lo)),0,3), 0 when
 * d*sc_lo is 0.  All in fp32, one rounding per operation, ties to even. */
void qso_q2k_quantize_rows(const float *w, int64_t n_rows, int64_t K, uint8_t *out) {
    int64_t nb = K / QSO_BLOCK_WEIGHTS;
    for (int64_t r = 0; r < n_rows; r++) {
        for (int64_t b = 0; b < nb; b++) {
            const float *x = w + r * K + b * QSO_BLOCK_WEIGHTS;
            float s[16], m[16], maxs = 0.0f, maxm = 0.0f;
            for (int sb = 0; sb < 16; sb++) {
                float mn = x[16 * sb], mx = x[16 * sb];
                for (int i = 1; i < 16; i++) {
                    float v = x[16 * sb + i];
                    if (v < mn) mn = v;
                    if (v > mx) mx = v;
                }
                m[sb] = mn < 0.0f ? -mn : 0.0f;
                s[sb] = (mx + m[sb]) / 3.0f;
                if (s[sb] > maxs) maxs = s[sb];
                if (m[sb] > maxm) maxm = m[sb];
            }
            uint16_t dh = qso_float_to_half(maxs / 15.0f);
            uint16_t mh = qso_float_to_half(maxm / 15.0f);
            float df = (float)qso_half_to_double(dh);
            float mf = (float)qso_half_to_double(mh);
            uint8_t sc[16], q[256];
            for (int sb = 0; sb < 16; sb++) {
                int lo = df > 0.0f ? (int)clampf_(rintf(s[sb] / df), 0.0f, 15.0f) : 0;
                int hi = mf > 0.0f ? (int)clampf_(rintf(m[sb] / mf), 0.0f, 15.0f) : 0;
                sc[sb] = (uint8_t)(lo | (hi << 4));
                float step = df * (float)lo;
                float base = mf * (float)hi;
                for (int i = 0; i < 16; i++) {
                    int qi = 0;
                    if (step > 0.0f) qi = (int)clampf_(rintf((x[16 * sb + i] + base) / step), 0.0f, 3.0f);
                    q[16 * sb + i] = (uint8_t)qi;
                }
            }
            qso_q2k_pack(sc, q, dh, mh, out + (r * nb + b) * QSO_BLOCK_BYTES);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Q4_K block (the 4-bit sibling format: routed experts of late layers)  */
/* ------------------------------------------------------------------ */

/* The pages name Q4_K experts (QuarkStar (q36) README, "Model Weights", the
 * Layers34-39Q4KExperts file) and say GGUF quant layouts are kept
 * ("Acknowledgements"); they do not spell the block out.  Reading, the GGUF
 * Q4_K layout, 144 bytes per 256 weights:
 *   d (fp16 LE, bytes 0-1) | dmin (fp16 LE, bytes 2-3) | scales[12] (bytes
 *   4-15) | qs[128] (bytes 16-143);
 *   eight 32-weight sub-blocks, each with a 6-bit scale sc and a 6-bit min m:
 *     j < 4:  sc = S[j] & 63,                          m = S[j+4] & 63
 *     j >= 4: sc = (S[j+4] & 15) | (S[j-4] >> 6) << 4, m = (S[j+4] >> 4) | (S[j] >> 6) << 4
 *   weight 64c + l (c in 0..3): l < 32 is the low nibble of qs[32c + l]
 *   (sub-block 2c), l >= 32 the high nibble of qs[32c + l - 32] (sub-block 2c+1);
 *   w = d * sc * q - dmin * m. */
#define QSO_Q4K_BYTES 144

void qso_q4k_unpack(const uint8_t *blk, uint8_t *sc, uint8_t *m, uint8_t *q, uint16_t *d, uint16_t *dmin) {
    const uint8_t *S = blk + 4;
    for (int j = 0; j < 8; j++) {
        if (j < 4) {
            sc[j] = (uint8_t)(S[j] & 63);
            m[j] = (uint8_t)(S[j + 4] & 63);
        } else {
            sc[j] = (uint8_t)((S[j + 4] & 15) | ((S[j - 4] >> 6) << 4));
            m[j] = (uint8_t)((S[j + 4] >> 4) | ((S[j] >> 6) << 4));
        }
    }
    for (int i = 0; i < QSO_BLOCK_WEIGHTS; i++) {
        int c = i / 64, l = i % 64;
        q[i] = (uint8_t)(l < 32 ? (blk[16 + 32 * c + l] & 15) : (blk[16 + 32 * c + l - 32] >> 4));
    }
    *d = (uint16_t)(blk[0] | (blk[1] << 8));
    *dmin = (uint16_t)(blk[2] | (blk[3] << 8));
}

/* Inverse of qso_q4k_unpack (sc, m in 0..63, q in 0..15). */
void qso_q4k_pack(const uint8_t *sc, const uint8_t *m, const uint8_t *q, uint16_t d, uint16_t dmin, uint8_t *blk) {
    memset(blk, 0, QSO_Q4K_BYTES);
    blk[0] = (uint8_t)(d & 0xff);
    blk[1] = (uint8_t)(d >> 8);
    blk[2] = (uint8_t)(dmin & 0xff);
    blk[3] = (uint8_t)(dmin >> 8);
    uint8_t *S = blk + 4;
    for (int j = 0; j < 4; j++) {
        S[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        S[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        S[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
    for (int i = 0; i < QSO_BLOCK_WEIGHTS; i++) {
        int c = i / 64, l = i % 64;
        if (l < 32) blk[16 + 32 * c + l] |= (uint8_t)(q[i] & 15);
        else blk[16 + 32 * c + l - 32] |= (uint8_t)((q[i] & 15) << 4);
    }
}

/* Decode one row of K weights (K/256 consecutive Q4_K blocks) to double, exactly. */
void qso_q4k_dequant_row(const uint8_t *row, int64_t K, double *w) {
    uint8_t sc[8], m[8], q[256];
    uint16_t dh, mh;
    for (int64_t b = 0; b < K / QSO_BLOCK_WEIGHTS; b++) {
        qso_q4k_unpack(row + b * QSO_Q4K_BYTES, sc, m, q, &dh, &mh);
        double d = qso_half_to_double(dh), dmin = qso_half_to_double(mh);
        for (int i = 0; i < QSO_BLOCK_WEIGHTS; i++) {
            int j = i / 32;
            w[b * QSO_BLOCK_WEIGHTS + i] = d * (double)sc[j] * (double)q[i] - dmin * (double)m[j];
        }
    }
}

void qso_q4k_dequant_rows(const uint8_t *rows, int64_t n_rows, int64_t K, double *w) {
    int64_t row_bytes = K / QSO_BLOCK_WEIGHTS * QSO_Q4K_BYTES;
    for (int64_t r = 0; r < n_rows; r++) qso_q4k_dequant_row(rows + r * row_bytes, K, w + r * K);
}

/* Round-to-nearest Q4_K encoder (set-up step, not part of the layer), the same
 * reading as the Q2_K one with 32-weight sub-blocks, 4-bit codes and 6-bit
 * scales: per sub-block m = max(0, -min w), s = (max w + m)/15; per block
 * d = fp16(max s / 63), dmin = fp16(max m / 63); sc = clamp(rint(s/d),0,63),
 * mc = clamp(rint(m/dmin),0,63) (0 when the divisor is 0);
 * q = clamp(rint((w + dmin*mc)/(d*sc)),0,15), 0 when d*sc is 0.  All in fp32,
 * one rounding per operation, ties to even. */
void qso_q4k_quantize_rows(const float *w, int64_t n_rows, int64_t K, uint8_t *out) {
    int64_t nb = K / QSO_BLOCK_WEIGHTS;
    for (int64_t r = 0; r < n_rows; r++) {
        for (int64_t b = 0; b < nb; b++) {
            const float *x = w + r * K + b * QSO_BLOCK_WEIGHTS;
            float s[8], mm[8], maxs = 0.0f, maxm = 0.0f;
            for (int j = 0; j < 8; j++) {
                float mn = x[32 * j], mx = x[32 * j];
                for (int i = 1; i < 32; i++) {
                    float v = x[32 * j + i];
                    if (v < mn) mn = v;
                    if (v > mx) mx = v;
                }
                mm[j] = mn < 0.0f ? -mn : 0.0f;
                s[j] = (mx + mm[j]) / 15.0f;
                if (s[j] > maxs) maxs = s[j];
                if (mm[j] > maxm) maxm = mm[j];
            }
            uint16_t dh = qso_float_to_half(maxs / 63.0f);
            uint16_t mh = qso_float_to_half(maxm / 63.0f);
            float df = (float)qso_half_to_double(dh);
            float mf = (float)qso_half_to_double(mh);
            uint8_t sc[8], mc[8], q[256];
            for (int j = 0; j < 8; j++) {
                int a = df > 0.0f ? (int)clampf_(rintf(s[j] / df), 0.0f, 63.0f) : 0;
                int c = mf > 0.0f ? (int)clampf_(rintf(mm[j] / mf), 0.0f, 63.0f) : 0;
                sc[j] = (uint8_t)a;
                mc[j] = (uint8_t)c;
                float step = df * (float)a;
                float base = mf * (float)c;
                for (int i = 0; i < 32; i++) {
                    int qi = 0;
                    if (step > 0.0f) qi = (int)clampf_(rintf((x[32 * j + i] + base) / step), 0.0f, 15.0f);
                    q[32 * j + i] = (uint8_t)qi;
                }
            }
            qso_q4k_pack(sc, mc, q, dh, mh, out + (r * nb + b) * QSO_Q4K_BYTES);
        }
    }
}

/* ------------------------------------------------------------------ */
/* the layer                                                            */
/* ------------------------------------------------------------------ */

#define QSO_X_F32 0
#define QSO_X_BF16 1

static void widen_x_(const void *x, int x_dtype, int64_t n, double *out) {
    if (x_dtype == QSO_X_BF16) {
        const uint16_t *b = (const uint16_t *)x;
        for (int64_t i = 0; i < n; i++) out[i] = qso_bf16_to_double(b[i]);
    } else {
        const float *f = (const float *)x;
        for (int64_t i = 0; i < n; i++) out[i] = (double)f[i];
    }
}

static double silu_(double z) { return z / (1.0 + exp(-z)); }
static double sigmoid_(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Router for T tokens: l = Wr x (+ b); ids = the k largest logits in
 * descending order, ties to the lower expert index; p = softmax over those k
 * logits; margin = l_(k) - l_(k+1) (+inf when k == E).  logits may be NULL. */
int qso_route(int H, int E, int k, int T, const void *x, int x_dtype, const float *Wr, const float *bias,
              int32_t *ids, double *p, double *margin, double *logits) {
    if (k < 1 || k > E) return 1;
    double *xw = (double *)malloc(sizeof(double) * (size_t)H);
    double *l = (double *)malloc(sizeof(double) * (size_t)E);
    int *ord = (int *)malloc(sizeof(int) * (size_t)E);
    if (!xw || !l || !ord) { free(xw); free(l); free(ord); return 2; }
    for (int t = 0; t < T; t++) {
        widen_x_((const char *)x + (size_t)t * H * (x_dtype == QSO_X_BF16 ? 2 : 4), x_dtype, H, xw);
        for (int e = 0; e < E; e++) {
            double acc = 0.0;
            for (int h = 0; h < H; h++) acc += (double)Wr[(size_t)e * H + h] * xw[h];
            if (bias) acc += (double)bias[e];
            l[e] = acc;
            if (logits) logits[(size_t)t * E + e] = acc;
        }
        /* insertion sort of expert indices by (logit descending, index ascending) */
        for (int e = 0; e < E; e++) {
            int j = e;
            while (j > 0 && l[ord[j - 1]] < l[e]) { ord[j] = ord[j - 1]; j--; }
            ord[j] = e;
        }
        double lmax = l[ord[0]], den = 0.0;
        for (int j = 0; j < k; j++) den += exp(l[ord[j]] - lmax);
        for (int j = 0; j < k; j++) {
            ids[(size_t)t * k + j] = ord[j];
            p[(size_t)t * k + j] = exp(l[ord[j]] - lmax) / den;
        }
        margin[t] = (k < E) ? l[ord[k - 1]] - l[ord[k]] : INFINITY;
    }
    free(xw); free(l); free(ord);
    return 0;
}

/* Grouping: counts per expert, exclusive offsets (E+1 entries), and perm =
 * the flat indices t*k+slot listed expert by expert, ascending inside each. */
void qso_group(int E, int k, int T, const int32_t *ids, int32_t *counts, int32_t *offsets, int32_t *perm) {
    int64_t n = (int64_t)T * k;
    for (int e = 0; e < E; e++) counts[e] = 0;
    for (int64_t i = 0; i < n; i++) counts[ids[i]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; e++) offsets[e + 1] = offsets[e] + counts[e];
    int64_t pos = 0;
    for (int e = 0; e < E; e++)
        for (int64_t i = 0; i < n; i++)
            if (ids[i] == e) perm[pos++] = (int32_t)i;
}

/* Expert weight formats: fmt 0 = Q2_K (84-byte blocks), 1 = Q4_K (144-byte blocks). */
#define QSO_FMT_Q2K 0
#define QSO_FMT_Q4K 1

static int64_t row_bytes_(int fmt, int64_t K) {
    return K / QSO_BLOCK_WEIGHTS * (fmt == QSO_FMT_Q4K ? QSO_Q4K_BYTES : QSO_BLOCK_BYTES);
}

static void dequant_row_(int fmt, const uint8_t *row, int64_t K, double *w) {
    if (fmt == QSO_FMT_Q4K) qso_q4k_dequant_row(row, K, w);
    else qso_q2k_dequant_row(row, K, w);
}

/* One routed expert on one widened token: h = silu(Wg x) * (Wu x).
 * blob = the expert's bytes in format fmt: gate rows [F x H], then up rows
 * [F x H], then down rows [H x F]; blocks run along each row. */
void qso_expert_gateup_fmt(int fmt, int H, int F, const uint8_t *blob, const double *x, double *h) {
    int64_t rb = row_bytes_(fmt, H);
    double *w = (double *)malloc(sizeof(double) * (size_t)H);
    for (int r = 0; r < F; r++) {
        double g = 0.0, u = 0.0;
        dequant_row_(fmt, blob + (int64_t)r * rb, H, w);
        for (int i = 0; i < H; i++) g += w[i] * x[i];
        dequant_row_(fmt, blob + (int64_t)(F + r) * rb, H, w);
        for (int i = 0; i < H; i++) u += w[i] * x[i];
        h[r] = silu_(g) * u;
    }
    free(w);
}

void qso_expert_gateup(int H, int F, const uint8_t *blob, const double *x, double *h) {
    qso_expert_gateup_fmt(QSO_FMT_Q2K, H, F, blob, x, h);
}

/* y = Wd h for one expert (down rows [H x F] after gate and up). */
void qso_expert_down_fmt(int fmt, int H, int F, const uint8_t *blob, const double *h, double *y) {
    int64_t rb_h = row_bytes_(fmt, H);
    int64_t rb_f = row_bytes_(fmt, F);
    const uint8_t *down = blob + 2 * (int64_t)F * rb_h;
    double *w = (double *)malloc(sizeof(double) * (size_t)F);
    for (int r = 0; r < H; r++) {
        double acc = 0.0;
        dequant_row_(fmt, down + (int64_t)r * rb_f, F, w);
        for (int i = 0; i < F; i++) acc += w[i] * h[i];
        y[r] = acc;
    }
    free(w);
}

void qso_expert_down(int H, int F, const uint8_t *blob, const double *h, double *y) {
    qso_expert_down_fmt(QSO_FMT_Q2K, H, F, blob, h, y);
}

/* Gated bf16 shared expert on one widened token:
 * g = sigmoid(w_sg . x), hs = silu(Wsg x) * (Wsu x), y = g * Wsd hs. */
void qso_shared_expert(int H, int S, const uint16_t *wg, const uint16_t *wu, const uint16_t *wd,
                       const uint16_t *wsig, const double *x, double *hs, double *gate, double *y) {
    double z = 0.0;
    for (int i = 0; i < H; i++) z += qso_bf16_to_double(wsig[i]) * x[i];
    *gate = sigmoid_(z);
    for (int r = 0; r < S; r++) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < H; i++) {
            g += qso_bf16_to_double(wg[(size_t)r * H + i]) * x[i];
            u += qso_bf16_to_double(wu[(size_t)r * H + i]) * x[i];
        }
        hs[r] = silu_(g) * u;
    }
    for (int r = 0; r < H; r++) {
        double acc = 0.0;
        for (int i = 0; i < S; i++) acc += qso_bf16_to_double(wd[(size_t)r * S + i]) * hs[i];
        y[r] = *gate * acc;
    }
}

/* The whole layer for tokens t0 .. t0+nt-1 of x (x points at token 0).
 * Outputs per token (all row-major, indexed by absolute token t):
 *   ids [T x k], p [T x k], margin [T], y [T x H]   (required)
 *   h [T*k x F] (SwiGLU of each (t, slot)), hs [T x S], gate [T]  (nullable)
 * S == 0 or wg == NULL skips the shared expert. */
int qso_moe_ffn_fmt(int fmt, int H, int E, int k, int F, int S, int t0, int nt, const void *x, int x_dtype,
                    const float *Wr, const float *bias, const uint8_t *experts, int64_t expert_stride,
                    const uint16_t *wg, const uint16_t *wu, const uint16_t *wd, const uint16_t *wsig,
                    int32_t *ids, double *p, double *margin, double *y, double *h_out, double *hs_out,
                    double *gate_out) {
    size_t xb = (size_t)H * (x_dtype == QSO_X_BF16 ? 2 : 4);
    double *xw = (double *)malloc(sizeof(double) * (size_t)H);
    double *h = (double *)malloc(sizeof(double) * (size_t)F);
    double *ye = (double *)malloc(sizeof(double) * (size_t)H);
    double *hs = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    if (!xw || !h || !ye || !hs) { free(xw); free(h); free(ye); free(hs); return 2; }
    int rc = 0;
    for (int t = t0; t < t0 + nt && rc == 0; t++) {
        const void *xt = (const char *)x + (size_t)t * xb;
        rc = qso_route(H, E, k, 1, xt, x_dtype, Wr, bias, ids + (size_t)t * k, p + (size_t)t * k, margin + t, NULL);
        if (rc) break;
        widen_x_(xt, x_dtype, H, xw);
        double *yt = y + (size_t)t * H;
        for (int i = 0; i < H; i++) yt[i] = 0.0;
        for (int j = 0; j < k; j++) {
            int e = ids[(size_t)t * k + j];
            const uint8_t *blob = experts + (int64_t)e * expert_stride;
            qso_expert_gateup_fmt(fmt, H, F, blob, xw, h);
            if (h_out) memcpy(h_out + ((size_t)t * k + j) * F, h, sizeof(double) * (size_t)F);
            qso_expert_down_fmt(fmt, H, F, blob, h, ye);
            for (int i = 0; i < H; i++) yt[i] += p[(size_t)t * k + j] * ye[i];
        }
        if (S > 0 && wg) {
            double g;
            qso_shared_expert(H, S, wg, wu, wd, wsig, xw, hs, &g, ye);
            for (int i = 0; i < H; i++) yt[i] += ye[i];
            if (hs_out) memcpy(hs_out + (size_t)t * S, hs, sizeof(double) * (size_t)S);
            if (gate_out) gate_out[t] = g;
        }
    }
    free(xw); free(h); free(ye); free(hs);
    return rc;
}

/* The layer with Q2_K experts (see qso_moe_ffn_fmt). */
int qso_moe_ffn(int H, int E, int k, int F, int S, int t0, int nt, const void *x, int x_dtype,
                const float *Wr, const float *bias, const uint8_t *experts, int64_t expert_stride,
                const uint16_t *wg, const uint16_t *wu, const uint16_t *wd, const uint16_t *wsig,
                int32_t *ids, double *p, double *margin, double *y, double *h_out, double *hs_out,
                double *gate_out) {
    return qso_moe_ffn_fmt(QSO_FMT_Q2K, H, E, k, F, S, t0, nt, x, x_dtype, Wr, bias, experts, expert_stride, wg, wu,
                           wd, wsig, ids, p, margin, y, h_out, hs_out, gate_out);
}

/* ------------------------------------------------------------------ */
/* directional steering of the FFN output                               */
/* ------------------------------------------------------------------ */

/* QuarkStar (q36) README, "Steering" (the same projection as DwarfStar's
 * "Steering" section): every token's FFN output row is edited in place as
 *     y <- y - scale * d * (d . y)
 * with d the layer's direction (stored normalised; this function does not
 * normalise it) and scale a scalar: positive removes the direction, negative
 * amplifies it, zero leaves y unchanged.  y: [T x H] double, d: [H] fp32
 * widened exactly.  The dot is taken first for the whole row, then the row
 * is updated, in the order of the formula. */
void qso_steer_rows(int H, int T, const float *d, double scale, double *y) {
    for (int t = 0; t < T; t++) {
        double *yt = y + (size_t)t * H;
        double c = 0.0;
        for (int i = 0; i < H; i++) c += (double)d[i] * yt[i];
        for (int i = 0; i < H; i++) yt[i] = yt[i] - scale * (double)d[i] * c;
    }
}

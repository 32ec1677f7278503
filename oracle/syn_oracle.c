/*
 * syn_oracle.c — plain, slow, scalar CPU oracle for GGUF block-quantized mul_mat.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path may link, load or call this
 * file; only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * Compiled with `-O2 -ffp-contract=off`: every float operation below is one IEEE-754
 * binary32 operation rounded to nearest even, in the order written.  Integer block
 * sums are exact.  The final product is accumulated in binary64 and rounded once.
 *
 * Sources (web pages the method is described on):
 *  - "The GGML ecosystem, and where synapse fits", section 5 "Quantization": the table
 *    of block formats (Q8_0 32 weights in 34 B, w = d*q; Q4_K 256 weights in 144 B,
 *    w = d*sc*q - dmin*m with 6-bit sc/m; Q6_K 256 weights in 210 B, 16 sub-blocks of 16
 *    with int8 scales and 6-bit quants in a 4-bit and a 2-bit plane; Q8_K 256 int8, float
 *    d, 16 int16 sub-block sums, activations only).
 *  - same page, "Products: weights against quantized activations": activations are
 *    converted to the weight type's vec_dot_type (Q8_0 for Q8_0, Q8_K for K-quants)
 *    once per row, and each weight block is dotted with the matching activation block
 *    in integer arithmetic; only the per-block scales are float.
 *  - yakaai ggml documentation, examples/simple: ggml_mul_mat(A, B^T) = C^T, i.e. the
 *    result holds, for each activation row t, the outputs of every weight row.
 *
 * Readings taken where the pages are silent (each one is listed in the design notes):
 *  - fp32 -> fp16 is round-to-nearest-even, written here from the IEEE-754 definition.
 *  - "round" is C roundf (ties away from zero).
 *  - Q8_0 codes are computed against the STORED fp16 scale D, not the fp32 d.
 *  - Q8_K keeps d = amax/127 in fp32; bsums[k] = sum of codes 16k..16k+15.
 *  - Q4_K: plain min-max encoder (per 32-sub-block range / 15, mins clamped to <= 0);
 *    super-scales d = fp16(max s / 63), dmin = fp16(max m / 63).
 *  - Q6_K: symmetric encoder, codes q' in [-32, 31] stored as q' + 32; d = fp16(max s/127).
 *  - Q4_0 / Q5_0 (same table: 32 weights, fp16 d, w = d*(q - 8) / d*(q - 16), q 4 / 5 bits):
 *    d = m / -8 (Q4_0) or m / -16 (Q5_0), m the block's value of largest magnitude with
 *    its sign, so that m itself maps to q = 0; q = clamp(round(x / D) + 8 (16), 0, 15 (31)).
 *  - F16 weights: one fp16 value per weight (RNE from fp32); their vec_dot_type is F16
 *    (the activations rounded to fp16 the same way); each product w*x is exact in fp64.
 *  - byte layout inside the blocks: the public GGUF on-disk layout (see the pack/unpack
 *    routines for the field order).
 *  - non-finite input, or a scale that overflows fp16, is rejected (status -5).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_Q8_0 1
#define ORC_Q4_K 2
#define ORC_Q6_K 3
#define ORC_Q8_K 4
#define ORC_Q4_0 5
#define ORC_Q5_0 6
#define ORC_F16 7

#define ORC_OK 0
#define ORC_ERR_TYPE (-1)
#define ORC_ERR_SHAPE (-2)
#define ORC_ERR_RANGE (-5)

/* ------------------------------------------------------------------------------------ */
/* binary16 <-> binary32, from the IEEE-754 definition                                   */
/* ------------------------------------------------------------------------------------ */

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* Round the non-negative integer m * 2^-s to an integer, ties to even (s may be <= 0). */
static uint64_t rne_shift(uint64_t m, int s) {
    if (s <= 0) return m << (-s);
    if (s >= 63) return 0; /* m < 2^25, so the value is far below one half */
    uint64_t q = m >> s;
    uint64_t r = m & ((1ull << s) - 1);
    uint64_t half = 1ull << (s - 1);
    if (r > half || (r == half && (q & 1))) q += 1;
    return q;
}

uint16_t orc_fp32_to_fp16(float f) {
    uint32_t u = f2u(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t e8 = (u >> 23) & 0xFFu;
    uint32_t frac = u & 0x7FFFFFu;
    if (e8 == 0xFFu) return frac ? (uint16_t)(sign | 0x7E00u) : (uint16_t)(sign | 0x7C00u);
    /* value = m * 2^e exactly, m < 2^24 */
    uint64_t m;
    int e;
    if (e8 == 0) { m = frac; e = -149; }
    else { m = (uint64_t)frac | 0x800000u; e = (int)e8 - 150; }
    if (m == 0) return sign;
    /* exponent of the leading bit: value in [2^E, 2^(E+1)) */
    int msb = 63 - __builtin_clzll(m);
    int E = e + msb;
    if (E < -14) {
        /* binary16 subnormal range: quantum 2^-24, result n in [0, 1024] */
        uint64_t n = rne_shift(m, -(e + 24));
        return (uint16_t)(sign | (uint16_t)n); /* n == 1024 encodes the smallest normal */
    }
    /* normal range: quantum 2^(E-10), significand n in [1024, 2048] */
    uint64_t n = rne_shift(m, (E - 10) - e);
    if (n == 2048) { n = 1024; E += 1; }
    if (E > 15) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(n - 1024));
}

float orc_fp16_to_fp32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e5 = (h >> 10) & 0x1Fu;
    uint32_t mant = h & 0x3FFu;
    float v;
    if (e5 == 0x1Fu) return u2f(sign | 0x7F800000u | (mant << 13));
    if (e5 == 0) v = ldexpf((float)mant, -24);
    else v = ldexpf((float)(mant + 1024u), (int)e5 - 25);
    return (sign ? -v : v);
}

void orc_fp32_to_fp16_array(const float* src, uint16_t* dst, int64_t n) {
    for (int64_t i = 0; i < n; i++) dst[i] = orc_fp32_to_fp16(src[i]);
}

void orc_fp16_to_fp32_array(const uint16_t* src, float* dst, int64_t n) {
    for (int64_t i = 0; i < n; i++) dst[i] = orc_fp16_to_fp32(src[i]);
}

/* ------------------------------------------------------------------------------------ */
/* format sizes                                                                          */
/* ------------------------------------------------------------------------------------ */

int64_t orc_block_elems(int type) {
    switch (type) {
    case ORC_Q8_0: case ORC_Q4_0: case ORC_Q5_0: return 32;
    case ORC_Q4_K: case ORC_Q6_K: case ORC_Q8_K: return 256;
    case ORC_F16: return 1;
    default: return -1;
    }
}

/* Q8_0: fp16 d + 32 int8.  Q4_K: fp16 d, fp16 dmin, 12 B scales, 128 B nibbles.
 * Q6_K: 128 B low 4 bits, 64 B high 2 bits, 16 int8 scales, fp16 d.
 * Q8_K: fp32 d, 256 int8, 16 int16 sums. */
int64_t orc_block_bytes(int type) {
    switch (type) {
    case ORC_Q8_0: return 2 + 32;
    case ORC_Q4_K: return 2 + 2 + 12 + 128;
    case ORC_Q6_K: return 128 + 64 + 16 + 2;
    case ORC_Q8_K: return 4 + 256 + 2 * 16;
    case ORC_Q4_0: return 2 + 16;
    case ORC_Q5_0: return 2 + 4 + 16;
    case ORC_F16: return 2;
    default: return -1;
    }
}

/* ------------------------------------------------------------------------------------ */
/* unpacked block representations                                                        */
/* ------------------------------------------------------------------------------------ */

typedef struct { uint16_t d; int8_t q[32]; } q8_0_u;
typedef struct { uint16_t d, dmin; uint8_t sc[8], mn[8]; uint8_t q[256]; } q4_k_u;  /* q in 0..15 */
typedef struct { uint16_t d; int8_t sc[16]; uint8_t q[256]; } q6_k_u;                /* q in 0..63 */
typedef struct { float d; int8_t q[256]; int16_t bsums[16]; } q8_k_u;
typedef struct { uint16_t d; uint8_t q[32]; } qx_0_u;  /* Q4_0: q in 0..15; Q5_0: q in 0..31 */

static float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* ---- Q8_0 ---- */

static int quant_q8_0(const float* x, q8_0_u* b) {
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        if (!isfinite(x[i])) return ORC_ERR_RANGE;
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    b->d = orc_fp32_to_fp16(d);
    if ((b->d & 0x7C00u) == 0x7C00u) return ORC_ERR_RANGE;
    float D = orc_fp16_to_fp32(b->d);
    for (int i = 0; i < 32; i++)
        b->q[i] = (D == 0.0f) ? 0 : (int8_t)clampf(roundf(x[i] / D), -127.0f, 127.0f);
    return ORC_OK;
}

static void pack_q8_0(const q8_0_u* b, uint8_t* p) {
    p[0] = (uint8_t)(b->d & 0xFF);
    p[1] = (uint8_t)(b->d >> 8);
    memcpy(p + 2, b->q, 32);
}

static void unpack_q8_0(const uint8_t* p, q8_0_u* b) {
    b->d = (uint16_t)(p[0] | (p[1] << 8));
    memcpy(b->q, p + 2, 32);
}

static void deq_q8_0(const q8_0_u* b, float* y) {
    float D = orc_fp16_to_fp32(b->d);
    for (int i = 0; i < 32; i++) y[i] = D * (float)b->q[i];
}

/* ---- Q8_K ---- */

static int quant_q8_k(const float* x, q8_k_u* b) {
    float amax = 0.0f;
    for (int i = 0; i < 256; i++) {
        if (!isfinite(x[i])) return ORC_ERR_RANGE;
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    b->d = d;
    for (int i = 0; i < 256; i++)
        b->q[i] = (d == 0.0f) ? 0 : (int8_t)clampf(roundf(x[i] / d), -127.0f, 127.0f);
    for (int k = 0; k < 16; k++) {
        int s = 0;
        for (int i = 0; i < 16; i++) s += b->q[16 * k + i];
        b->bsums[k] = (int16_t)s;
    }
    return ORC_OK;
}

static void pack_q8_k(const q8_k_u* b, uint8_t* p) {
    memcpy(p, &b->d, 4);   /* little-endian binary32 */
    memcpy(p + 4, b->q, 256);
    for (int k = 0; k < 16; k++) {
        uint16_t v = (uint16_t)b->bsums[k];
        p[260 + 2 * k] = (uint8_t)(v & 0xFF);
        p[260 + 2 * k + 1] = (uint8_t)(v >> 8);
    }
}

static void unpack_q8_k(const uint8_t* p, q8_k_u* b) {
    memcpy(&b->d, p, 4);
    memcpy(b->q, p + 4, 256);
    for (int k = 0; k < 16; k++)
        b->bsums[k] = (int16_t)(uint16_t)(p[260 + 2 * k] | (p[260 + 2 * k + 1] << 8));
}

static void deq_q8_k(const q8_k_u* b, float* y) {
    for (int i = 0; i < 256; i++) y[i] = b->d * (float)b->q[i];
}

/* ---- Q4_K ---- */

static int quant_q4_k(const float* x, q4_k_u* b) {
    float s[8], m[8];
    float smax = 0.0f, mmax = 0.0f;
    for (int i = 0; i < 256; i++)
        if (!isfinite(x[i])) return ORC_ERR_RANGE;
    for (int j = 0; j < 8; j++) {
        const float* xj = x + 32 * j;
        float lo = 0.0f, hi = xj[0];
        for (int i = 0; i < 32; i++) {
            if (xj[i] < lo) lo = xj[i];
            if (xj[i] > hi) hi = xj[i];
        }
        s[j] = (hi - lo) / 15.0f;
        m[j] = (lo < 0.0f) ? -lo : 0.0f;
        if (s[j] > smax) smax = s[j];
        if (m[j] > mmax) mmax = m[j];
    }
    b->d = orc_fp32_to_fp16(smax / 63.0f);
    b->dmin = orc_fp32_to_fp16(mmax / 63.0f);
    if ((b->d & 0x7C00u) == 0x7C00u || (b->dmin & 0x7C00u) == 0x7C00u) return ORC_ERR_RANGE;
    float D = orc_fp16_to_fp32(b->d), Dm = orc_fp16_to_fp32(b->dmin);
    for (int j = 0; j < 8; j++) {
        b->sc[j] = (D == 0.0f) ? 0 : (uint8_t)fminf(63.0f, roundf(s[j] / D));
        b->mn[j] = (Dm == 0.0f) ? 0 : (uint8_t)fminf(63.0f, roundf(m[j] / Dm));
        float S = D * (float)b->sc[j];
        float M = Dm * (float)b->mn[j];
        for (int i = 0; i < 32; i++) {
            float xi = x[32 * j + i];
            b->q[32 * j + i] = (S > 0.0f) ? (uint8_t)clampf(roundf((xi + M) / S), 0.0f, 15.0f) : 0;
        }
    }
    return ORC_OK;
}

/* Scale bytes: 0..3 hold sc0..sc3 (low 6 bits) and the top 2 bits of sc4..sc7;
 * 4..7 hold mn0..mn3 (low 6 bits) and the top 2 bits of mn4..mn7;
 * 8..11 hold the low 4 bits of sc4..sc7 (low nibble) and of mn4..mn7 (high nibble).
 * Codes: byte 32c+l holds sub-block 2c element l (low nibble), 2c+1 element l (high). */
static void pack_q4_k(const q4_k_u* b, uint8_t* p) {
    p[0] = (uint8_t)(b->d & 0xFF); p[1] = (uint8_t)(b->d >> 8);
    p[2] = (uint8_t)(b->dmin & 0xFF); p[3] = (uint8_t)(b->dmin >> 8);
    uint8_t* sb = p + 4;
    for (int j = 0; j < 4; j++) {
        sb[j] = (uint8_t)((b->sc[j] & 63) | ((b->sc[j + 4] >> 4) << 6));
        sb[j + 4] = (uint8_t)((b->mn[j] & 63) | ((b->mn[j + 4] >> 4) << 6));
        sb[j + 8] = (uint8_t)((b->sc[j + 4] & 15) | ((b->mn[j + 4] & 15) << 4));
    }
    uint8_t* qs = p + 16;
    for (int c = 0; c < 4; c++)
        for (int l = 0; l < 32; l++)
            qs[32 * c + l] = (uint8_t)(b->q[64 * c + l] | (b->q[64 * c + 32 + l] << 4));
}

static void unpack_q4_k(const uint8_t* p, q4_k_u* b) {
    b->d = (uint16_t)(p[0] | (p[1] << 8));
    b->dmin = (uint16_t)(p[2] | (p[3] << 8));
    const uint8_t* sb = p + 4;
    for (int j = 0; j < 4; j++) {
        b->sc[j] = sb[j] & 63;
        b->mn[j] = sb[j + 4] & 63;
        b->sc[j + 4] = (uint8_t)((sb[j + 8] & 15) | ((sb[j] >> 6) << 4));
        b->mn[j + 4] = (uint8_t)((sb[j + 8] >> 4) | ((sb[j + 4] >> 6) << 4));
    }
    const uint8_t* qs = p + 16;
    for (int c = 0; c < 4; c++)
        for (int l = 0; l < 32; l++) {
            b->q[64 * c + l] = qs[32 * c + l] & 15;
            b->q[64 * c + 32 + l] = qs[32 * c + l] >> 4;
        }
}

static void deq_q4_k(const q4_k_u* b, float* y) {
    float D = orc_fp16_to_fp32(b->d), Dm = orc_fp16_to_fp32(b->dmin);
    for (int j = 0; j < 8; j++) {
        float S = D * (float)b->sc[j];
        float M = Dm * (float)b->mn[j];
        for (int i = 0; i < 32; i++) y[32 * j + i] = S * (float)b->q[32 * j + i] - M;
    }
}

/* ---- Q6_K ---- */

static int quant_q6_k(const float* x, q6_k_u* b) {
    float s[16];
    float smax = 0.0f;
    for (int i = 0; i < 256; i++)
        if (!isfinite(x[i])) return ORC_ERR_RANGE;
    for (int j = 0; j < 16; j++) {
        float amax = 0.0f;
        for (int i = 0; i < 16; i++) {
            float a = fabsf(x[16 * j + i]);
            if (a > amax) amax = a;
        }
        s[j] = amax / 31.0f;
        if (s[j] > smax) smax = s[j];
    }
    b->d = orc_fp32_to_fp16(smax / 127.0f);
    if ((b->d & 0x7C00u) == 0x7C00u) return ORC_ERR_RANGE;
    float D = orc_fp16_to_fp32(b->d);
    for (int j = 0; j < 16; j++) {
        b->sc[j] = (D == 0.0f) ? 0 : (int8_t)fminf(127.0f, roundf(s[j] / D));
        float S = D * (float)b->sc[j];
        for (int i = 0; i < 16; i++) {
            float xi = x[16 * j + i];
            int qq = (S > 0.0f) ? (int)clampf(roundf(xi / S), -32.0f, 31.0f) : 0;
            b->q[16 * j + i] = (uint8_t)(qq + 32);
        }
    }
    return ORC_OK;
}

/* Within each 128-weight half h and lane l < 32, weights l, l+32, l+64, l+96 of the half
 * take their low 4 bits from: low nibble of ql[64h+l], low nibble of ql[64h+l+32],
 * high nibble of ql[64h+l], high nibble of ql[64h+l+32]; and their top 2 bits from
 * qh[32h+l] bits 0-1, 2-3, 4-5, 6-7.  scales[j] belongs to weights 16j..16j+15. */
static void pack_q6_k(const q6_k_u* b, uint8_t* p) {
    uint8_t* ql = p;
    uint8_t* qh = p + 128;
    for (int h = 0; h < 2; h++)
        for (int l = 0; l < 32; l++) {
            const uint8_t* q = b->q + 128 * h;
            uint8_t q1 = q[l], q2 = q[l + 32], q3 = q[l + 64], q4 = q[l + 96];
            ql[64 * h + l] = (uint8_t)((q1 & 15) | ((q3 & 15) << 4));
            ql[64 * h + l + 32] = (uint8_t)((q2 & 15) | ((q4 & 15) << 4));
            qh[32 * h + l] = (uint8_t)((q1 >> 4) | ((q2 >> 4) << 2) | ((q3 >> 4) << 4) | ((q4 >> 4) << 6));
        }
    memcpy(p + 192, b->sc, 16);
    p[208] = (uint8_t)(b->d & 0xFF);
    p[209] = (uint8_t)(b->d >> 8);
}

static void unpack_q6_k(const uint8_t* p, q6_k_u* b) {
    const uint8_t* ql = p;
    const uint8_t* qh = p + 128;
    for (int h = 0; h < 2; h++)
        for (int l = 0; l < 32; l++) {
            uint8_t* q = b->q + 128 * h;
            uint8_t a = ql[64 * h + l], c = ql[64 * h + l + 32], hb = qh[32 * h + l];
            q[l] = (uint8_t)((a & 15) | ((hb & 3) << 4));
            q[l + 32] = (uint8_t)((c & 15) | (((hb >> 2) & 3) << 4));
            q[l + 64] = (uint8_t)((a >> 4) | (((hb >> 4) & 3) << 4));
            q[l + 96] = (uint8_t)((c >> 4) | (((hb >> 6) & 3) << 4));
        }
    memcpy(b->sc, p + 192, 16);
    b->d = (uint16_t)(p[208] | (p[209] << 8));
}

static void deq_q6_k(const q6_k_u* b, float* y) {
    float D = orc_fp16_to_fp32(b->d);
    for (int j = 0; j < 16; j++) {
        float S = D * (float)b->sc[j];
        for (int i = 0; i < 16; i++) y[16 * j + i] = S * (float)((int)b->q[16 * j + i] - 32);
    }
}

/* ------------------------------------------------------------------------------------ */
/* row-level quantize / dequantize                                                       */
/* ------------------------------------------------------------------------------------ */

/* ---- Q4_0 / Q5_0: 32 weights, w = D * (q - off), off = 8 (4-bit) or 16 (5-bit) ---- */

static int quant_qx_0(const float* x, qx_0_u* b, int off) {
    float m = 0.0f, amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        if (!isfinite(x[i])) return ORC_ERR_RANGE;
        float a = fabsf(x[i]);
        if (a > amax) { amax = a; m = x[i]; }
    }
    float d = m / -(float)off;
    b->d = orc_fp32_to_fp16(d);
    if ((b->d & 0x7C00u) == 0x7C00u) return ORC_ERR_RANGE;
    float D = orc_fp16_to_fp32(b->d);
    for (int i = 0; i < 32; i++)
        b->q[i] = (D == 0.0f) ? (uint8_t)off
                              : (uint8_t)clampf(roundf(x[i] / D) + (float)off, 0.0f, (float)(2 * off - 1));
    return ORC_OK;
}

/* Q4_0 bytes: d, then qs[16]: byte l holds q[l] (low nibble) and q[l + 16] (high nibble). */
static void pack_q4_0(const qx_0_u* b, uint8_t* p) {
    p[0] = (uint8_t)(b->d & 0xFF);
    p[1] = (uint8_t)(b->d >> 8);
    for (int l = 0; l < 16; l++) p[2 + l] = (uint8_t)((b->q[l] & 15) | ((b->q[l + 16] & 15) << 4));
}

static void unpack_q4_0(const uint8_t* p, qx_0_u* b) {
    b->d = (uint16_t)(p[0] | (p[1] << 8));
    for (int l = 0; l < 16; l++) {
        b->q[l] = p[2 + l] & 15;
        b->q[l + 16] = p[2 + l] >> 4;
    }
}

/* Q5_0 bytes: d, then qh (32 bits, little endian: bit i = the fifth bit of q[i]), then
 * qs[16] holding the low four bits as in Q4_0. */
static void pack_q5_0(const qx_0_u* b, uint8_t* p) {
    p[0] = (uint8_t)(b->d & 0xFF);
    p[1] = (uint8_t)(b->d >> 8);
    uint32_t qh = 0;
    for (int i = 0; i < 32; i++) qh |= (uint32_t)((b->q[i] >> 4) & 1) << i;
    for (int k = 0; k < 4; k++) p[2 + k] = (uint8_t)(qh >> (8 * k));
    for (int l = 0; l < 16; l++) p[6 + l] = (uint8_t)((b->q[l] & 15) | ((b->q[l + 16] & 15) << 4));
}

static void unpack_q5_0(const uint8_t* p, qx_0_u* b) {
    b->d = (uint16_t)(p[0] | (p[1] << 8));
    uint32_t qh = (uint32_t)p[2] | ((uint32_t)p[3] << 8) | ((uint32_t)p[4] << 16) | ((uint32_t)p[5] << 24);
    for (int l = 0; l < 16; l++) {
        b->q[l] = (uint8_t)((p[6 + l] & 15) | (((qh >> l) & 1) << 4));
        b->q[l + 16] = (uint8_t)((p[6 + l] >> 4) | (((qh >> (l + 16)) & 1) << 4));
    }
}

static void deq_qx_0(const qx_0_u* b, int off, float* y) {
    float D = orc_fp16_to_fp32(b->d);
    for (int i = 0; i < 32; i++) y[i] = D * (float)((int)b->q[i] - off);
}

static int check_shape(int type, int64_t n_rows, int64_t n_per_row) {
    int64_t be = orc_block_elems(type);
    if (be < 0) return ORC_ERR_TYPE;
    if (n_rows < 0 || n_per_row <= 0 || n_per_row % be) return ORC_ERR_SHAPE;
    return ORC_OK;
}

int orc_quantize(int type, const float* src, uint8_t* dst, int64_t n_rows, int64_t n_per_row) {
    int st = check_shape(type, n_rows, n_per_row);
    if (st) return st;
    int64_t be = orc_block_elems(type), bb = orc_block_bytes(type);
    int64_t nb = n_rows * (n_per_row / be);
    for (int64_t k = 0; k < nb; k++) {
        const float* x = src + k * be;
        uint8_t* p = dst + k * bb;
        switch (type) {
        case ORC_Q8_0: { q8_0_u b; if ((st = quant_q8_0(x, &b))) return st; pack_q8_0(&b, p); break; }
        case ORC_Q8_K: { q8_k_u b; if ((st = quant_q8_k(x, &b))) return st; pack_q8_k(&b, p); break; }
        case ORC_Q4_K: { q4_k_u b; if ((st = quant_q4_k(x, &b))) return st; pack_q4_k(&b, p); break; }
        case ORC_Q6_K: { q6_k_u b; if ((st = quant_q6_k(x, &b))) return st; pack_q6_k(&b, p); break; }
        case ORC_Q4_0: { qx_0_u b; if ((st = quant_qx_0(x, &b, 8))) return st; pack_q4_0(&b, p); break; }
        case ORC_Q5_0: { qx_0_u b; if ((st = quant_qx_0(x, &b, 16))) return st; pack_q5_0(&b, p); break; }
        case ORC_F16: {
            if (!isfinite(x[0])) return ORC_ERR_RANGE;
            uint16_t h = orc_fp32_to_fp16(x[0]);
            if ((h & 0x7C00u) == 0x7C00u) return ORC_ERR_RANGE;  /* overflow to infinity */
            p[0] = (uint8_t)(h & 0xFF); p[1] = (uint8_t)(h >> 8);
            break;
        }
        }
    }
    return ORC_OK;
}

int orc_dequantize(int type, const uint8_t* src, float* dst, int64_t n_rows, int64_t n_per_row) {
    int st = check_shape(type, n_rows, n_per_row);
    if (st) return st;
    int64_t be = orc_block_elems(type), bb = orc_block_bytes(type);
    int64_t nb = n_rows * (n_per_row / be);
    for (int64_t k = 0; k < nb; k++) {
        const uint8_t* p = src + k * bb;
        float* y = dst + k * be;
        switch (type) {
        case ORC_Q8_0: { q8_0_u b; unpack_q8_0(p, &b); deq_q8_0(&b, y); break; }
        case ORC_Q8_K: { q8_k_u b; unpack_q8_k(p, &b); deq_q8_k(&b, y); break; }
        case ORC_Q4_K: { q4_k_u b; unpack_q4_k(p, &b); deq_q4_k(&b, y); break; }
        case ORC_Q6_K: { q6_k_u b; unpack_q6_k(p, &b); deq_q6_k(&b, y); break; }
        case ORC_Q4_0: { qx_0_u b; unpack_q4_0(p, &b); deq_qx_0(&b, 8, y); break; }
        case ORC_Q5_0: { qx_0_u b; unpack_q5_0(p, &b); deq_qx_0(&b, 16, y); break; }
        case ORC_F16: y[0] = orc_fp16_to_fp32((uint16_t)(p[0] | (p[1] << 8))); break;
        }
    }
    return ORC_OK;
}

/* Field-level views, so that tests can check codes and scales against the formulas. */
int orc_unpack_q4_k(const uint8_t* p, uint16_t* d, uint16_t* dmin, uint8_t* sc, uint8_t* mn, uint8_t* q) {
    q4_k_u b; unpack_q4_k(p, &b);
    *d = b.d; *dmin = b.dmin; memcpy(sc, b.sc, 8); memcpy(mn, b.mn, 8); memcpy(q, b.q, 256);
    return ORC_OK;
}

int orc_unpack_qx_0(int type, const uint8_t* p, uint16_t* d, uint8_t* q) {
    qx_0_u b;
    if (type == ORC_Q4_0) unpack_q4_0(p, &b);
    else if (type == ORC_Q5_0) unpack_q5_0(p, &b);
    else return ORC_ERR_TYPE;
    *d = b.d; memcpy(q, b.q, 32);
    return ORC_OK;
}

int orc_unpack_q6_k(const uint8_t* p, uint16_t* d, int8_t* sc, uint8_t* q) {
    q6_k_u b; unpack_q6_k(p, &b);
    *d = b.d; memcpy(sc, b.sc, 16); memcpy(q, b.q, 256);
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------ */
/* integer block sums and the product                                                    */
/* ------------------------------------------------------------------------------------ */

/* vec_dot_type of a weight format: Q8_0 for Q8_0, Q4_0 and Q5_0, Q8_K for the K-quants. */
static int vec_dot_type(int wtype) {
    switch (wtype) {
    case ORC_Q8_0: case ORC_Q4_0: case ORC_Q5_0: return ORC_Q8_0;
    case ORC_Q4_K: case ORC_Q6_K: return ORC_Q8_K;
    case ORC_F16: return ORC_F16;
    default: return -1;
    }
}

int orc_vec_dot_type(int wtype) { return vec_dot_type(wtype); }

/* Integer sums of one (weight block, activation block) pair.
 *  Q8_0: I  = sum_i qw_i * qx_i                                       -> s[0] = I
 *  Q4_K: A  = sum_j sc_j * sum_{i in j} q_i * qx_i                    -> s[0] = A
 *        Bm = sum_j mn_j * (bsum_{2j} + bsum_{2j+1})                  -> s[1] = Bm
 *  Q6_K: C  = sum_j sc_j * sum_{i in j} (q_i - 32) * qx_i             -> s[0] = C
 *  Q4_0 / Q5_0: I = sum_i (q_i - 8 / 16) * qx_i                       -> s[0] = I */
static void block_sums(int wtype, const uint8_t* wp, const uint8_t* xp, int32_t s[2]) {
    s[0] = 0; s[1] = 0;
    if (wtype == ORC_Q8_0) {
        q8_0_u w, x; unpack_q8_0(wp, &w); unpack_q8_0(xp, &x);
        int32_t I = 0;
        for (int i = 0; i < 32; i++) I += (int32_t)w.q[i] * (int32_t)x.q[i];
        s[0] = I;
    } else if (wtype == ORC_Q4_K) {
        q4_k_u w; q8_k_u x; unpack_q4_k(wp, &w); unpack_q8_k(xp, &x);
        int32_t A = 0, Bm = 0;
        for (int j = 0; j < 8; j++) {
            int32_t dot = 0;
            for (int i = 32 * j; i < 32 * j + 32; i++) dot += (int32_t)w.q[i] * (int32_t)x.q[i];
            A += (int32_t)w.sc[j] * dot;
            Bm += (int32_t)w.mn[j] * ((int32_t)x.bsums[2 * j] + (int32_t)x.bsums[2 * j + 1]);
        }
        s[0] = A; s[1] = Bm;
    } else if (wtype == ORC_Q6_K) {
        q6_k_u w; q8_k_u x; unpack_q6_k(wp, &w); unpack_q8_k(xp, &x);
        int32_t C = 0;
        for (int j = 0; j < 16; j++) {
            int32_t dot = 0;
            for (int i = 16 * j; i < 16 * j + 16; i++) dot += ((int32_t)w.q[i] - 32) * (int32_t)x.q[i];
            C += (int32_t)w.sc[j] * dot;
        }
        s[0] = C;
    } else if (wtype == ORC_Q4_0 || wtype == ORC_Q5_0) {
        qx_0_u w; q8_0_u x;
        int off = wtype == ORC_Q4_0 ? 8 : 16;
        if (wtype == ORC_Q4_0) unpack_q4_0(wp, &w); else unpack_q5_0(wp, &w);
        unpack_q8_0(xp, &x);
        int32_t I = 0;
        for (int i = 0; i < 32; i++) I += ((int32_t)w.q[i] - off) * (int32_t)x.q[i];
        s[0] = I;
    }
}

/* fp64 contribution of one block pair:
 *  Q8_0, Q4_0, Q5_0: D_w * D_x * I;   Q4_K: D * d_x * A - Dm * d_x * Bm;   Q6_K: D * d_x * C. */
static double block_value(int wtype, const uint8_t* wp, const uint8_t* xp, const int32_t s[2]) {
    if (wtype == ORC_Q8_0 || wtype == ORC_Q4_0 || wtype == ORC_Q5_0) {
        double Dw = orc_fp16_to_fp32((uint16_t)(wp[0] | (wp[1] << 8)));
        double Dx = orc_fp16_to_fp32((uint16_t)(xp[0] | (xp[1] << 8)));
        return Dw * Dx * (double)s[0];
    }
    float dxf; memcpy(&dxf, xp, 4);
    double dx = dxf;
    if (wtype == ORC_Q4_K) {
        double D = orc_fp16_to_fp32((uint16_t)(wp[0] | (wp[1] << 8)));
        double Dm = orc_fp16_to_fp32((uint16_t)(wp[2] | (wp[3] << 8)));
        return D * dx * (double)s[0] - Dm * dx * (double)s[1];
    }
    double D = orc_fp16_to_fp32((uint16_t)(wp[208] | (wp[209] << 8)));
    return D * dx * (double)s[0];
}

/* Block sums for every (token t, row o, block b): S[((t*n_out + o)*nb + b)*2 + {0,1}].
 * Xq holds n_tok rows already in the vec_dot_type of wtype. */
int orc_block_sums(int wtype, const uint8_t* W, int64_t n_out, int64_t n_in,
                   const uint8_t* Xq, int64_t n_tok, int32_t* S) {
    int xt = vec_dot_type(wtype);
    if (xt < 0 || wtype == ORC_F16) return ORC_ERR_TYPE;  /* F16 products are not integer */
    int st = check_shape(wtype, n_out, n_in);
    if (st) return st;
    int64_t nb = n_in / orc_block_elems(wtype);
    int64_t wb = orc_block_bytes(wtype), xb = orc_block_bytes(xt);
    for (int64_t t = 0; t < n_tok; t++)
        for (int64_t o = 0; o < n_out; o++)
            for (int64_t b = 0; b < nb; b++)
                block_sums(wtype, W + (o * nb + b) * wb, Xq + (t * nb + b) * xb,
                           S + ((t * n_out + o) * nb + b) * 2);
    return ORC_OK;
}

/* y[t][o] for one (o, t) pair: fp64 sum over blocks, rounded once to fp32. */
static float dot_row(int wtype, const uint8_t* Wrow, const uint8_t* Xrow, int64_t nb, int64_t wb, int64_t xb) {
    double acc = 0.0;
    if (wtype == ORC_F16) {  /* exact fp16 x fp16 products, summed in fp64 */
        for (int64_t i = 0; i < nb; i++) {
            double w = orc_fp16_to_fp32((uint16_t)(Wrow[2 * i] | (Wrow[2 * i + 1] << 8)));
            double x = orc_fp16_to_fp32((uint16_t)(Xrow[2 * i] | (Xrow[2 * i + 1] << 8)));
            acc += w * x;
        }
        return (float)acc;
    }
    for (int64_t b = 0; b < nb; b++) {
        int32_t s[2];
        block_sums(wtype, Wrow + b * wb, Xrow + b * xb, s);
        acc += block_value(wtype, Wrow + b * wb, Xrow + b * xb, s);
    }
    return (float)acc;
}

typedef struct {
    int wtype; const uint8_t* W; int64_t n_out, n_in; const uint8_t* Xq; int64_t n_tok; float* Y;
    int64_t o0, o1;
} mm_job;

static void* mm_worker(void* arg) {
    mm_job* j = (mm_job*)arg;
    int xt = vec_dot_type(j->wtype);
    int64_t nb = j->n_in / orc_block_elems(j->wtype);
    int64_t wb = orc_block_bytes(j->wtype), xb = orc_block_bytes(xt);
    for (int64_t t = 0; t < j->n_tok; t++)
        for (int64_t o = j->o0; o < j->o1; o++)
            j->Y[t * j->n_out + o] = dot_row(j->wtype, j->W + o * nb * wb, j->Xq + t * nb * xb, nb, wb, xb);
    return NULL;
}

/* ggml_mul_mat(W, X) with W n_out x n_in (rows contiguous) in a weight format and X
 * n_tok x n_in fp32: X is first quantized to the vec_dot_type, row by row; then
 * Y[t*n_out + o] = sum_b blockvalue(W[o, b], Xq[t, b]).  n_threads splits the rows. */
int orc_mul_mat(int wtype, const uint8_t* W, int64_t n_out, int64_t n_in,
                const float* X, int64_t n_tok, float* Y, int n_threads) {
    int xt = vec_dot_type(wtype);
    if (xt < 0) return ORC_ERR_TYPE;
    int st = check_shape(wtype, n_out, n_in);
    if (st) return st;
    if (n_tok < 0) return ORC_ERR_SHAPE;
    int64_t xrow = (n_in / orc_block_elems(xt)) * orc_block_bytes(xt);
    uint8_t* Xq = (uint8_t*)malloc((size_t)(xrow * (n_tok > 0 ? n_tok : 1)));
    if (!Xq) return ORC_ERR_SHAPE;
    st = orc_quantize(xt, X, Xq, n_tok, n_in);
    if (st) { free(Xq); return st; }
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if (n_threads > n_out) n_threads = (int)n_out;
    mm_job jobs[256];
    pthread_t th[256];
    for (int k = 0; k < n_threads; k++) {
        jobs[k] = (mm_job){wtype, W, n_out, n_in, Xq, n_tok, Y,
                           n_out * k / n_threads, n_out * (k + 1) / n_threads};
        if (n_threads > 1) pthread_create(&th[k], NULL, mm_worker, &jobs[k]);
        else mm_worker(&jobs[k]);
    }
    if (n_threads > 1)
        for (int k = 0; k < n_threads; k++) pthread_join(th[k], NULL);
    free(Xq);
    return ORC_OK;
}

/* The same product evaluated only at the listed (row, token) pairs:
 * Ys[i*n_rows_s + r] = Y[toks[i]][rows[r]]. */
int orc_mul_mat_sampled(int wtype, const uint8_t* W, int64_t n_out, int64_t n_in,
                        const float* X, int64_t n_tok,
                        const int64_t* rows, int64_t n_rows_s, const int64_t* toks, int64_t n_toks_s,
                        float* Ys) {
    int xt = vec_dot_type(wtype);
    if (xt < 0) return ORC_ERR_TYPE;
    int st = check_shape(wtype, n_out, n_in);
    if (st) return st;
    int64_t nb = n_in / orc_block_elems(wtype);
    int64_t wb = orc_block_bytes(wtype), xb = orc_block_bytes(xt);
    uint8_t* xq = (uint8_t*)malloc((size_t)(nb * xb));
    if (!xq) return ORC_ERR_SHAPE;
    for (int64_t i = 0; i < n_toks_s; i++) {
        int64_t t = toks[i];
        if (t < 0 || t >= n_tok) { free(xq); return ORC_ERR_SHAPE; }
        st = orc_quantize(xt, X + t * n_in, xq, 1, n_in);
        if (st) { free(xq); return st; }
        for (int64_t r = 0; r < n_rows_s; r++) {
            int64_t o = rows[r];
            if (o < 0 || o >= n_out) { free(xq); return ORC_ERR_SHAPE; }
            Ys[i * n_rows_s + r] = dot_row(wtype, W + o * nb * wb, xq, nb, wb, xb);
        }
    }
    free(xq);
    return ORC_OK;
}

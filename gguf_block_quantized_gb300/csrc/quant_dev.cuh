// quant_dev.cuh — warp-cooperative block encoders, used by the quantize kernels and by
// the activation step of the product kernels (the same code, so that the activations a
// product uses are exactly those syn_quantize_activations returns).
//
// Encoders: plain readings of the format table in "The GGML ecosystem, and where synapse
// fits", section 5, with the activation conversion of "Products: weights against
// quantized activations" (Q8_0 for Q8_0 weights, Q8_K for the K-quants).  Every float
// operation is an explicit round-to-nearest intrinsic: no contraction into FMA, IEEE
// division, so the bytes equal those of a scalar fp32 implementation.
#pragma once
#include "common.cuh"

namespace syn {

__device__ __forceinline__ float clampf(float v, float lo, float hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

__device__ __forceinline__ uint32_t pack4_s8(int a, int b, int c, int d) {
    return (uint32_t)(a & 0xFF) | ((uint32_t)(b & 0xFF) << 8) | ((uint32_t)(c & 0xFF) << 16) |
           ((uint32_t)(d & 0xFF) << 24);
}

template <int W>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int o = 1; o < W; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int W>
__device__ __forceinline__ float group_min(float v) {
#pragma unroll
    for (int o = 1; o < W; o <<= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ bool all_finite4(const float* v) {
    return isfinite(v[0]) && isfinite(v[1]) && isfinite(v[2]) && isfinite(v[3]);
}

// Codes q[i] = clamp(roundf(v[i] / d), -127, 127) (IEEE quotient, ties away from zero; a zero
// code as +0, a NaN quotient as 0, the integer an IEEE-to-integer conversion of it gives on the
// device), for d > 0 with |v[i] / d| below 2^21.  The product v * (1/d), with the reciprocal
// rounded once, lies within 3 * 2^-24 (relative) of the IEEE quotient, so where it is farther
// than 2^-12 from every half-integer both round to the same integer, taken here by adding and
// subtracting 1.5 * 2^23 (integer spacing at that magnitude).  A lane with any value nearer a
// half-integer, or non-finite, takes the IEEE division for all of its values.  Keeps the
// special-function and conversion pipes free of per-value divisions, roundings and conversions.
// CLAMP: the quotients may exceed 127.5 (the Q8_0 scale is rounded to fp16).
template <int N, bool CLAMP>
__device__ __forceinline__ void round_quots(const float* v, float d, float* q) {
    const float inv = __frcp_rn(d);
    bool ok = true;
#pragma unroll
    for (int i = 0; i < N; i++) {
        const float r = __fmul_rn(v[i], inv);
        const float n = __fsub_rn(__fadd_rn(r, 12582912.0f), 12582912.0f);
        ok = ok && fabsf(__fsub_rn(r, n)) < 0.5f - 1.0f / 4096.0f;
        q[i] = CLAMP ? clampf(n, -127.0f, 127.0f) : n;
    }
    if (!ok) {
#pragma unroll
        for (int i = 0; i < N; i++) {
            const float e = roundf(__fdiv_rn(v[i], d));
            q[i] = e == e ? __fadd_rn(clampf(e, -127.0f, 127.0f), 0.0f) : 0.0f;
        }
    }
}

// The integer value of a float holding an integer of magnitude below 2^22, without a
// conversion instruction (the low mantissa bits of q + 1.5 * 2^23).
__device__ __forceinline__ int int_of(float q) {
    return __float_as_int(__fadd_rn(q, 12582912.0f)) - 0x4B400000;
}

// ---------------------------------------------------------------------------------------
// Q8_0: groups of 8 lanes, 4 consecutive values per lane, one 32-block per group.
// Returns the 4 codes packed in a word and the stored scale (fp16 bits in *dbits).
// ---------------------------------------------------------------------------------------
// The codes as floats (exact integers, zero as +0); returns the fp16 scale bits.
__device__ __forceinline__ uint16_t q8_0_group_codes(const float v[4], float q[4]) {
    const float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    const float amax = group_max<8>(a);
    const __half hd = __float2half_rn(__fdiv_rn(amax, 127.0f));
    const float D = __half2float(hd);
    if (D == 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; i++) q[i] = 0.0f;
    } else {
        round_quots<4, true>(v, D, q);
    }
    return __half_as_ushort(hd);
}

__device__ __forceinline__ uint32_t q8_0_group(const float v[4], uint16_t* dbits,
                                               bool* finite) {
    float q[4];
    *dbits = q8_0_group_codes(v, q);
    *finite = all_finite4(v) && !__hisinf(__ushort_as_half(*dbits));
    return pack4_s8(int_of(q[0]), int_of(q[1]), int_of(q[2]), int_of(q[3]));
}

// ---------------------------------------------------------------------------------------
// Q4_0 / Q5_0 (OFF = 8 / 16): groups of 8 lanes, 4 consecutive values per lane, one
// 32-block per group.  m = the first value of largest magnitude (index order), d = m/-OFF,
// q = clamp(round(x/D) + OFF, 0, 2*OFF - 1).  Returns the 4 codes as bytes of a word.
// ---------------------------------------------------------------------------------------
template <int OFF>
__device__ __forceinline__ uint32_t qx_0_group(const float v[4], uint16_t* dbits, bool* finite) {
    const int e = threadIdx.x & 7;
    float a = 0.0f, m = 0.0f;
    int idx = 4 * e;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float ai = fabsf(v[i]);
        if (ai > a) { a = ai; m = v[i]; idx = 4 * e + i; }
    }
    // (largest magnitude, lowest index) over the 8 lanes of the group
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        const float ao = __shfl_xor_sync(0xffffffffu, a, o);
        const float mo = __shfl_xor_sync(0xffffffffu, m, o);
        const int io = __shfl_xor_sync(0xffffffffu, idx, o);
        if (ao > a || (ao == a && io < idx)) { a = ao; m = mo; idx = io; }
    }
    const float d = __fdiv_rn(m, -(float)OFF);
    const __half hd = __float2half_rn(d);
    const float D = __half2float(hd);
    int q[4];
#pragma unroll
    for (int i = 0; i < 4; i++)
        q[i] = (D == 0.0f) ? OFF
                           : (int)clampf(__fadd_rn(roundf(__fdiv_rn(v[i], D)), (float)OFF), 0.0f, (float)(2 * OFF - 1));
    *dbits = __half_as_ushort(hd);
    *finite = all_finite4(v) && !__hisinf(hd);
    return pack4_s8(q[0], q[1], q[2], q[3]);
}

// ---------------------------------------------------------------------------------------
// Q8_K: one warp per 256-block, 8 consecutive values per lane (lane L: 8L..8L+7).
// Returns the codes as two words, the fp32 scale, and in *bsum the sum of the 16 codes
// of sub-block L/2 (valid in every lane).
// ---------------------------------------------------------------------------------------
// The codes as floats (exact integers, zero as +0); returns d.  |v[i] / d| <= 127 up to
// rounding: no clamp on the fast path.
__device__ __forceinline__ float q8_k_warp_codes(const float v[8], float q[8]) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) a = fmaxf(a, fabsf(v[i]));
    const float amax = group_max<32>(a);
    const float d = __fdiv_rn(amax, 127.0f);
    if (d == 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; i++) q[i] = 0.0f;
    } else {
        round_quots<8, false>(v, d, q);
    }
    return d;
}

__device__ __forceinline__ void q8_k_warp(const float v[8], uint32_t* w0, uint32_t* w1,
                                          float* dout, int* bsum, bool* finite) {
    float qf[8];
    const float d = q8_k_warp_codes(v, qf);
    int q[8];
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        q[i] = int_of(qf[i]);
        s += q[i];
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    *w0 = pack4_s8(q[0], q[1], q[2], q[3]);
    *w1 = pack4_s8(q[4], q[5], q[6], q[7]);
    *dout = d;
    *bsum = s;
    *finite = all_finite4(v) && all_finite4(v + 4);
}

// ---------------------------------------------------------------------------------------
// Q4_K: one warp per 256-block, lane L holds values 8L..8L+7 (sub-block L/4).
// Produces the codes (two words, one nibble value per byte), the sub-block scale and
// min codes of the lane's sub-block, and the two fp16 super-scales.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void q4_k_warp(const float v[8], uint32_t* w0, uint32_t* w1,
                                          int* sc_out, int* mn_out, uint16_t* dbits,
                                          uint16_t* dminbits, bool* finite) {
    float lo = 0.0f, hi = v[0];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        lo = fminf(lo, v[i]);
        hi = fmaxf(hi, v[i]);
    }
    lo = group_min<4>(lo);
    hi = group_max<4>(hi);
    float s = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
    float m = (lo < 0.0f) ? -lo : 0.0f;
    // max over the warp; adding +0 turns a -0 maximum (all sub-blocks -0) into +0, the
    // value a scalar running maximum started at +0 keeps.
    float smax = __fadd_rn(group_max<32>(s), 0.0f);
    float mmax = group_max<32>(m);
    __half hd = __float2half_rn(__fdiv_rn(smax, 63.0f));
    __half hdm = __float2half_rn(__fdiv_rn(mmax, 63.0f));
    float D = __half2float(hd), Dm = __half2float(hdm);
    int sc = (D == 0.0f) ? 0 : (int)fminf(63.0f, roundf(__fdiv_rn(s, D)));
    int mn = (Dm == 0.0f) ? 0 : (int)fminf(63.0f, roundf(__fdiv_rn(m, Dm)));
    float S = __fmul_rn(D, (float)sc);
    float M = __fmul_rn(Dm, (float)mn);
    int q[8];
#pragma unroll
    for (int i = 0; i < 8; i++)
        q[i] = (S > 0.0f) ? (int)clampf(roundf(__fdiv_rn(__fadd_rn(v[i], M), S)), 0.0f, 15.0f) : 0;
    *w0 = pack4_s8(q[0], q[1], q[2], q[3]);
    *w1 = pack4_s8(q[4], q[5], q[6], q[7]);
    *sc_out = sc;
    *mn_out = mn;
    *dbits = __half_as_ushort(hd);
    *dminbits = __half_as_ushort(hdm);
    bool f = all_finite4(v) && all_finite4(v + 4);
    *finite = f && !__hisinf(hd) && !__hisinf(hdm);
}

// ---------------------------------------------------------------------------------------
// Q6_K: one warp per 256-block, lane L holds values 8L..8L+7 (sub-block L/2).
// Produces the stored codes q'+32 (0..63, one per byte), the lane's sub-block scale and
// the fp16 super-scale.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void q6_k_warp(const float v[8], uint32_t* w0, uint32_t* w1,
                                          int* sc_out, uint16_t* dbits, bool* finite) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) a = fmaxf(a, fabsf(v[i]));
    float amax = group_max<2>(a);
    float s = __fdiv_rn(amax, 31.0f);
    float smax = group_max<32>(s);
    __half hd = __float2half_rn(__fdiv_rn(smax, 127.0f));
    float D = __half2float(hd);
    int sc = (D == 0.0f) ? 0 : (int)fminf(127.0f, roundf(__fdiv_rn(s, D)));
    float S = __fmul_rn(D, (float)sc);
    int q[8];
#pragma unroll
    for (int i = 0; i < 8; i++)
        q[i] = ((S > 0.0f) ? (int)clampf(roundf(__fdiv_rn(v[i], S)), -32.0f, 31.0f) : 0) + 32;
    *w0 = pack4_s8(q[0], q[1], q[2], q[3]);
    *w1 = pack4_s8(q[4], q[5], q[6], q[7]);
    *sc_out = sc;
    *dbits = __half_as_ushort(hd);
    *finite = all_finite4(v) && all_finite4(v + 4) && !__hisinf(hd);
}

}  // namespace syn

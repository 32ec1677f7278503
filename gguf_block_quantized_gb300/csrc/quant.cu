// quant.cu — quantize / dequantize kernels, the stand-alone activation step, the prefill
// activation step (fp16 operand for the tensor cores) and the integer block sums.
//
// "The GGML ecosystem, and where synapse fits", section 5: block formats (format table),
// dequantize_row_* (embedding / norm expansion) and the activation conversion to the
// vec_dot_type ("Products: weights against quantized activations").
#include <atomic>

#include "kernels.h"
#include "quant_dev.cuh"

namespace syn {

// ---------------------------------------------------------------------------------------
// weight / block quantize: one warp per block (Q8_0: one warp per 4 blocks)
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ void st_u16(uint8_t* p, uint32_t v) {
    *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(v);
}

template <int T>
__global__ void __launch_bounds__(256) k_quantize(const float* __restrict__ src,
                                                  uint8_t* __restrict__ dst, int64_t n_blocks,
                                                  int* __restrict__ range_err) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    bool ok_all = true;
    if (T == SYN_Q4_0 || T == SYN_Q5_0) {
        // 4 blocks per warp step: lanes 8g..8g+7 own block 4*step+g, 4 values each
        constexpr int OFF = T == SYN_Q4_0 ? 8 : 16, BB = T == SYN_Q4_0 ? 18 : 22, QS = T == SYN_Q4_0 ? 2 : 6;
        for (int64_t base = warp * 4; base < n_blocks; base += n_warps * 4) {
            int64_t b = base + (lane >> 3);
            const int e = lane & 7;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (b < n_blocks) {
                float4 x = *reinterpret_cast<const float4*>(src + b * 32 + 4 * e);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            }
            uint16_t db;
            bool fin;
            const uint32_t q = qx_0_group<OFF>(v, &db, &fin);
            // byte l of the codes: q[l] in the low nibble, q[l + 16] in the high one; lanes
            // e < 4 hold q[4e..4e+3], lanes e + 4 hold q[16 + 4e ..]
            const uint32_t up = __shfl_down_sync(0xffffffffu, q, 4);
            uint32_t hb = 0;  // fifth bits of this lane's 4 codes at bits 4e..4e+3 (Q5_0)
            if (T == SYN_Q5_0) {
                const uint32_t t = (q >> 4) & 0x01010101u;
                hb = ((t | (t >> 7) | (t >> 14) | (t >> 21)) & 15u) << (4 * e);
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) hb |= __shfl_xor_sync(0xffffffffu, hb, o);
            }
            if (b < n_blocks) {
                uint8_t* p = dst + b * BB;
                if (e == 0) st_u16(p, db);
                if (T == SYN_Q5_0 && e == 0) {
                    st_u16(p + 2, hb & 0xFFFF);
                    st_u16(p + 4, hb >> 16);
                }
                if (e < 4) {
                    const uint32_t packed = (q & 0x0F0F0F0Fu) | ((up & 0x0F0F0F0Fu) << 4);
                    st_u16(p + QS + 4 * e, packed & 0xFFFF);
                    st_u16(p + QS + 4 * e + 2, packed >> 16);
                }
                ok_all &= fin;
            }
        }
    } else if (T == SYN_Q8_0) {
        // 4 blocks per warp step: lanes 8g..8g+7 own block 4*step+g
        for (int64_t base = warp * 4; base < n_blocks; base += n_warps * 4) {
            int64_t b = base + (lane >> 3);
            int e = (lane & 7) * 4;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (b < n_blocks) {
                float4 x = *reinterpret_cast<const float4*>(src + b * 32 + e);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            }
            uint16_t db;
            bool fin;
            uint32_t q = q8_0_group(v, &db, &fin);
            if (b < n_blocks) {
                uint8_t* p = dst + b * 34;
                if ((lane & 7) == 0) st_u16(p, db);
                st_u16(p + 2 + e, q & 0xFFFF);
                st_u16(p + 4 + e, q >> 16);
                ok_all &= fin;
            }
        }
    } else {
        for (int64_t b = warp; b < n_blocks; b += n_warps) {
            if (!SYN_IN_BOUNDS(b >= 0 && b < n_blocks)) break;
            const float* x = src + b * 256 + lane * 8;
            float4 x0 = *reinterpret_cast<const float4*>(x);
            float4 x1 = *reinterpret_cast<const float4*>(x + 4);
            float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            uint32_t w0, w1;
            bool fin;
            if (T == SYN_Q8_K) {
                float d;
                int bs;
                q8_k_warp(v, &w0, &w1, &d, &bs, &fin);
                uint8_t* p = dst + b * 292;
                if (lane == 0) *reinterpret_cast<float*>(p) = d;
                *reinterpret_cast<uint32_t*>(p + 4 + lane * 8) = w0;
                *reinterpret_cast<uint32_t*>(p + 8 + lane * 8) = w1;
                if ((lane & 1) == 0) st_u16(p + 260 + lane, (uint32_t)bs);
            } else if (T == SYN_Q4_K) {
                int sc, mn;
                uint16_t db, dmb;
                q4_k_warp(v, &w0, &w1, &sc, &mn, &db, &dmb, &fin);
                uint8_t* p = dst + b * 144;
                // codes: byte 32c+l = q[64c+l] | q[64c+32+l] << 4; lane L holds
                // q[8L..8L+7]; lanes with (L & 4) == 0 take the high nibbles from L+4.
                uint32_t h0 = __shfl_down_sync(0xffffffffu, w0, 4);
                uint32_t h1 = __shfl_down_sync(0xffffffffu, w1, 4);
                if ((lane & 4) == 0) {
                    int c = lane >> 3, l = (lane & 3) * 8;
                    uint2 out;
                    out.x = w0 | (h0 << 4);
                    out.y = w1 | (h1 << 4);
                    *reinterpret_cast<uint2*>(p + 16 + 32 * c + l) = out;
                }
                // 6-bit scales and mins: sub-block j's values sit in lane 4j
                int scj[8], mnj[8];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    scj[j] = __shfl_sync(0xffffffffu, sc, 4 * j);
                    mnj[j] = __shfl_sync(0xffffffffu, mn, 4 * j);
                }
                if (lane == 0) {
                    uint8_t sb[12];
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        sb[j] = (uint8_t)((scj[j] & 63) | ((scj[j + 4] >> 4) << 6));
                        sb[j + 4] = (uint8_t)((mnj[j] & 63) | ((mnj[j + 4] >> 4) << 6));
                        sb[j + 8] = (uint8_t)((scj[j + 4] & 15) | ((mnj[j + 4] & 15) << 4));
                    }
                    uint4 hdr;
                    hdr.x = (uint32_t)db | ((uint32_t)dmb << 16);
                    hdr.y = sb[0] | (sb[1] << 8) | (sb[2] << 16) | ((uint32_t)sb[3] << 24);
                    hdr.z = sb[4] | (sb[5] << 8) | (sb[6] << 16) | ((uint32_t)sb[7] << 24);
                    hdr.w = sb[8] | (sb[9] << 8) | (sb[10] << 16) | ((uint32_t)sb[11] << 24);
                    *reinterpret_cast<uint4*>(p) = hdr;
                }
            } else {  // Q6_K
                int sc;
                uint16_t db;
                q6_k_warp(v, &w0, &w1, &sc, &db, &fin);
                uint8_t* p = dst + b * 210;
                // lane L: half h = L/16, quarter = (L%16)/4, l0 = 8*(L%4).  Quarter-0
                // lanes gather quarters 1..3 (lanes +4, +8, +12) and write the planes.
                uint32_t b0 = __shfl_down_sync(0xffffffffu, w0, 4), b1 = __shfl_down_sync(0xffffffffu, w1, 4);
                uint32_t c0 = __shfl_down_sync(0xffffffffu, w0, 8), c1 = __shfl_down_sync(0xffffffffu, w1, 8);
                uint32_t d0 = __shfl_down_sync(0xffffffffu, w0, 12), d1 = __shfl_down_sync(0xffffffffu, w1, 12);
                if ((lane & 15) < 4) {
                    int h = lane >> 4, l0 = (lane & 3) * 8;
                    uint32_t qa[2] = {w0, w1}, qb[2] = {b0, b1}, qc[2] = {c0, c1}, qd[2] = {d0, d1};
#pragma unroll
                    for (int k = 0; k < 2; k++) {
                        uint32_t lo1 = (qa[k] & 0x0F0F0F0Fu) | ((qc[k] & 0x0F0F0F0Fu) << 4);
                        uint32_t lo2 = (qb[k] & 0x0F0F0F0Fu) | ((qd[k] & 0x0F0F0F0Fu) << 4);
                        uint32_t hb = ((qa[k] >> 4) & 0x03030303u) | (((qb[k] >> 4) & 0x03030303u) << 2) |
                                      (((qc[k] >> 4) & 0x03030303u) << 4) | (((qd[k] >> 4) & 0x03030303u) << 6);
                        uint8_t* ql = p + 64 * h + l0 + 4 * k;
                        uint8_t* qh = p + 128 + 32 * h + l0 + 4 * k;
                        st_u16(ql, lo1 & 0xFFFF); st_u16(ql + 2, lo1 >> 16);
                        st_u16(ql + 32, lo2 & 0xFFFF); st_u16(ql + 34, lo2 >> 16);
                        st_u16(qh, hb & 0xFFFF); st_u16(qh + 2, hb >> 16);
                    }
                }
                if ((lane & 1) == 0) p[192 + (lane >> 1)] = (uint8_t)(int8_t)sc;
                if (lane == 0) st_u16(p + 208, db);
            }
            ok_all &= fin;
        }
    }
    if (!__all_sync(0xffffffffu, ok_all) && lane == 0) atomicExch(range_err, 1);
}

// ---------------------------------------------------------------------------------------
// dequantize: one warp per block (Q8_0: one warp per 4 blocks), 8 outputs per lane
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ uint16_t ld_u16(const uint8_t* p) {
    return *reinterpret_cast<const uint16_t*>(p);
}

template <int T>
__global__ void __launch_bounds__(256) k_dequantize(const uint8_t* __restrict__ src,
                                                    float* __restrict__ dst, int64_t n_blocks) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    if (T == SYN_Q4_0 || T == SYN_Q5_0) {
        constexpr int OFF = T == SYN_Q4_0 ? 8 : 16, BB = T == SYN_Q4_0 ? 18 : 22, QS = T == SYN_Q4_0 ? 2 : 6;
        for (int64_t base = warp * 4; base < n_blocks; base += n_warps * 4) {
            int64_t b = base + (lane >> 3);
            if (b >= n_blocks) continue;
            const uint8_t* p = src + b * BB;
            const float D = h2f_bits(ld_u16(p));
            const int e = (lane & 7) * 4;  // values e .. e+3
            const int l = e & 15, sh = e >= 16 ? 4 : 0;
            uint32_t qh = 0;
            if (T == SYN_Q5_0) qh = (uint32_t)ld_u16(p + 2) | ((uint32_t)ld_u16(p + 4) << 16);
            float y[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                int q = (p[QS + l + i] >> sh) & 15;
                if (T == SYN_Q5_0) q |= (int)((qh >> (e + i)) & 1) << 4;
                y[i] = __fmul_rn(D, (float)(q - OFF));
            }
            *reinterpret_cast<float4*>(dst + b * 32 + e) = make_float4(y[0], y[1], y[2], y[3]);
        }
        return;
    }
    if (T == SYN_Q8_0) {
        for (int64_t base = warp * 4; base < n_blocks; base += n_warps * 4) {
            int64_t b = base + (lane >> 3);
            if (b >= n_blocks) continue;
            const uint8_t* p = src + b * 34;
            float D = h2f_bits(ld_u16(p));
            int e = (lane & 7) * 4;
            float4 y;
            y.x = __fmul_rn(D, (float)(int8_t)p[2 + e]);
            y.y = __fmul_rn(D, (float)(int8_t)p[3 + e]);
            y.z = __fmul_rn(D, (float)(int8_t)p[4 + e]);
            y.w = __fmul_rn(D, (float)(int8_t)p[5 + e]);
            *reinterpret_cast<float4*>(dst + b * 32 + e) = y;
        }
        return;
    }
    for (int64_t b = warp; b < n_blocks; b += n_warps) {
        if (!SYN_IN_BOUNDS(b >= 0 && b < n_blocks)) break;
        float y[8];
        if (T == SYN_Q8_K) {
            const uint8_t* p = src + b * 292;
            float d = *reinterpret_cast<const float*>(p);
            uint32_t w0 = *reinterpret_cast<const uint32_t*>(p + 4 + lane * 8);
            uint32_t w1 = *reinterpret_cast<const uint32_t*>(p + 8 + lane * 8);
#pragma unroll
            for (int i = 0; i < 4; i++) {
                y[i] = __fmul_rn(d, (float)(int8_t)(w0 >> (8 * i)));
                y[4 + i] = __fmul_rn(d, (float)(int8_t)(w1 >> (8 * i)));
            }
        } else if (T == SYN_Q4_K) {
            const uint8_t* p = src + b * 144;
            float D = h2f_bits(ld_u16(p)), Dm = h2f_bits(ld_u16(p + 2));
            const uint8_t* sb = p + 4;
            int j = lane >> 2;  // sub-block of this lane's 8 values
            int sc, mn;
            if (j < 4) {
                sc = sb[j] & 63;
                mn = sb[j + 4] & 63;
            } else {
                sc = (sb[j + 4] & 15) | ((sb[j - 4] >> 6) << 4);
                mn = (sb[j + 4] >> 4) | ((sb[j] >> 6) << 4);
            }
            float S = __fmul_rn(D, (float)sc), M = __fmul_rn(Dm, (float)mn);
            int c = j >> 1, shift = (j & 1) * 4, l = (lane & 3) * 8;
            const uint8_t* qs = p + 16 + 32 * c + l;
#pragma unroll
            for (int i = 0; i < 8; i++) y[i] = __fsub_rn(__fmul_rn(S, (float)((qs[i] >> shift) & 15)), M);
        } else {  // Q6_K
            const uint8_t* p = src + b * 210;
            float D = h2f_bits(ld_u16(p + 208));
            int e0 = lane * 8;  // values e0..e0+7, one sub-block
            float S = __fmul_rn(D, (float)(int8_t)p[192 + (e0 >> 4)]);
            int h = e0 >> 7, w = e0 & 127, quarter = w >> 5, l0 = w & 31;
            const uint8_t* ql = p + 64 * h + l0 + ((quarter & 1) ? 32 : 0);
            const uint8_t* qh = p + 128 + 32 * h + l0;
            int nshift = (quarter >= 2) ? 4 : 0;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                int q = ((ql[i] >> nshift) & 15) | (((qh[i] >> (2 * quarter)) & 3) << 4);
                y[i] = __fmul_rn(S, (float)(q - 32));
            }
        }
        float* o = dst + b * 256 + lane * 8;
        *reinterpret_cast<float4*>(o) = make_float4(y[0], y[1], y[2], y[3]);
        *reinterpret_cast<float4*>(o + 4) = make_float4(y[4], y[5], y[6], y[7]);
    }
}

// ---------------------------------------------------------------------------------------
// K-quant weights -> fp16 rows (the prefill's A operand, expanded once per call): each value
// is the fp32 dequantization above (the same operations, so bit for bit the value
// syn_dequantize returns) rounded once to fp16.  One warp per 256-value block, 8 values per
// lane, one 16-byte store per lane; codes turned into floats by placing them in the low
// mantissa bits of 2^23 and subtracting it (exact), not by conversion instructions.
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ float code_f(uint32_t bytes, int i) {
    return __fsub_rn(__int_as_float((int)__byte_perm(bytes, 0x4B000000u, 0x7540u | (uint32_t)i)), 8388608.0f);
}

// The loads of a lane's share of one block, issued for DEQ_U blocks before any is expanded
// (the loop is bound by load latency otherwise).
struct DeqLoad {
    uint4 a;   // Q4_K: the 16-byte header; Q6_K: x = D bits, y = the sub-block scale byte
    uint2 q;   // Q4_K: 8 code bytes; Q6_K: 8 low-nibble bytes
    uint2 h;   // Q6_K: 8 high-bit bytes
};

template <int T>
__device__ __forceinline__ DeqLoad deq_load(const uint8_t* __restrict__ src, int64_t b, int lane) {
    DeqLoad L;
    if (T == SYN_Q4_K) {
        const uint8_t* p = src + b * 144;
        const int j = lane >> 2;
        L.a = *reinterpret_cast<const uint4*>(p);
        L.q = *reinterpret_cast<const uint2*>(p + 16 + 32 * (j >> 1) + 8 * (lane & 3));
        L.h = make_uint2(0, 0);
    } else {  // Q6_K: 2-byte aligned blocks, 16-bit loads
        const uint8_t* p = src + b * 210;
        const int h = lane >> 4, w = (lane * 8) & 127, quarter = w >> 5, l0 = w & 31;
        const uint8_t* ql = p + 64 * h + l0 + ((quarter & 1) ? 32 : 0);
        const uint8_t* qh = p + 128 + 32 * h + l0;
        L.a = make_uint4(ld_u16(p + 208), p[192 + (lane >> 1)], 0, 0);
        L.q = make_uint2((uint32_t)ld_u16(ql) | ((uint32_t)ld_u16(ql + 2) << 16),
                         (uint32_t)ld_u16(ql + 4) | ((uint32_t)ld_u16(ql + 6) << 16));
        L.h = make_uint2((uint32_t)ld_u16(qh) | ((uint32_t)ld_u16(qh + 2) << 16),
                         (uint32_t)ld_u16(qh + 4) | ((uint32_t)ld_u16(qh + 6) << 16));
    }
    return L;
}

template <int T>
__device__ __forceinline__ uint4 deq_expand(const DeqLoad& L, int lane) {
    float y[8];
    if (T == SYN_Q4_K) {
        // lane: values 8L .. 8L+7 of sub-block j = L/4 (code chunk j/2, nibble j%2)
        const float D = h2f_bits(L.a.x & 0xFFFF), Dm = h2f_bits(L.a.x >> 16);
        const int j = lane >> 2;
        // 6-bit scale and min of sub-block j from the 12 bytes after d and dmin
        const uint32_t sc_lo = L.a.y & 0x3F3F3F3Fu, mn_lo = L.a.z & 0x3F3F3F3Fu;
        const uint32_t sc_hi = (L.a.w & 0x0F0F0F0Fu) | ((L.a.y >> 2) & 0x30303030u);
        const uint32_t mn_hi = ((L.a.w >> 4) & 0x0F0F0F0Fu) | ((L.a.z >> 2) & 0x30303030u);
        const uint32_t sel = 0x4440u | (uint32_t)(j & 3);
        const int sc = (int)__byte_perm(j < 4 ? sc_lo : sc_hi, 0, sel);
        const int mn = (int)__byte_perm(j < 4 ? mn_lo : mn_hi, 0, sel);
        const float S = __fmul_rn(D, (float)sc), M = __fmul_rn(Dm, (float)mn);
        const int sh = (j & 1) * 4;
        const uint32_t v0 = (L.q.x >> sh) & 0x0F0F0F0Fu, v1 = (L.q.y >> sh) & 0x0F0F0F0Fu;
        // S * q is exact (S has at most 17 significant bits, q 4): one rounding, as in
        // the fp32 dequantization's multiply-then-subtract
#pragma unroll
        for (int i = 0; i < 4; i++) {
            y[i] = __fmaf_rn(S, code_f(v0, i), -M);
            y[4 + i] = __fmaf_rn(S, code_f(v1, i), -M);
        }
    } else {  // Q6_K: lane values 8L .. 8L+7, sub-block L/2
        const float S = __fmul_rn(h2f_bits((uint16_t)L.a.x), (float)(int8_t)(uint8_t)L.a.y);
        const int quarter = ((lane * 8) & 127) >> 5;
        const int ns = quarter >= 2 ? 4 : 0, hs = 2 * quarter;
        // the 6-bit codes q, one per byte; the value is S * (q - 32)
        const uint32_t c0 = ((L.q.x >> ns) & 0x0F0F0F0Fu) | (((L.h.x >> hs) & 0x03030303u) << 4);
        const uint32_t c1 = ((L.q.y >> ns) & 0x0F0F0F0Fu) | (((L.h.y >> hs) & 0x03030303u) << 4);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            y[i] = __fmul_rn(S, __fsub_rn(code_f(c0, i), 32.0f));
            y[4 + i] = __fmul_rn(S, __fsub_rn(code_f(c1, i), 32.0f));
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const __half2 h2 = __floats2half2_rn(y[2 * k], y[2 * k + 1]);
        o[k] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

constexpr int DEQ_U = 4;  // blocks per warp per iteration

template <int T>
__global__ void __launch_bounds__(256) k_deq_half(const uint8_t* __restrict__ src, __half* __restrict__ dst,
                                                  int64_t n_blocks) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t b0 = warp * DEQ_U; b0 < n_blocks; b0 += n_warps * DEQ_U) {
        DeqLoad L[DEQ_U];
#pragma unroll
        for (int u = 0; u < DEQ_U; u++)
            if (b0 + u < n_blocks) L[u] = deq_load<T>(src, b0 + u, lane);
#pragma unroll
        for (int u = 0; u < DEQ_U; u++)
            if (b0 + u < n_blocks && SYN_IN_BOUNDS(b0 + u >= 0))
                *reinterpret_cast<uint4*>(dst + (b0 + u) * 256 + lane * 8) = deq_expand<T>(L[u], lane);
    }
}

// ---------------------------------------------------------------------------------------
// activations -> vec_dot_type, structure-of-arrays (codes, scales, 16-sums)
// ---------------------------------------------------------------------------------------

template <int XT>
__global__ void __launch_bounds__(256) k_quantize_act(const float* __restrict__ X, int64_t n_rows_blocks,
                                                      int8_t* __restrict__ qs, float* __restrict__ d,
                                                      int16_t* __restrict__ bsums) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    if (XT == SYN_Q8_0) {
        for (int64_t base = warp * 4; base < n_rows_blocks; base += n_warps * 4) {
            int64_t b = base + (lane >> 3);
            int e = (lane & 7) * 4;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (b < n_rows_blocks) {
                float4 x = *reinterpret_cast<const float4*>(X + b * 32 + e);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            }
            uint16_t db;
            bool fin;
            uint32_t q = q8_0_group(v, &db, &fin);
            if (b < n_rows_blocks) {
                *reinterpret_cast<uint32_t*>(qs + b * 32 + e) = q;
                if ((lane & 7) == 0) d[b] = h2f_bits(db);
            }
        }
    } else {
        for (int64_t b = warp; b < n_rows_blocks; b += n_warps) {
            const float* x = X + b * 256 + lane * 8;
            float4 x0 = *reinterpret_cast<const float4*>(x);
            float4 x1 = *reinterpret_cast<const float4*>(x + 4);
            float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            uint32_t w0, w1;
            float dd;
            int bs;
            bool fin;
            q8_k_warp(v, &w0, &w1, &dd, &bs, &fin);
            *reinterpret_cast<uint2*>(qs + b * 256 + lane * 8) = make_uint2(w0, w1);
            if (lane == 0) d[b] = dd;
            if ((lane & 1) == 0 && bsums) bsums[b * 16 + (lane >> 1)] = (int16_t)bs;
        }
    }
}

// ---------------------------------------------------------------------------------------
// prefill activation step: quantize to the vec_dot_type and write x_hat = fp16(d * q),
// the tensor-core operand (token-major, n_in contiguous fp16 per token)
// ---------------------------------------------------------------------------------------

template <int XT>
__global__ void __launch_bounds__(256) k_act_half(const float* __restrict__ X, int64_t n_rows_blocks,
                                                  __half* __restrict__ xh) {
    // the product kernel that follows is launched as this kernel's programmatic dependent
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    // each warp loads its next blocks before it encodes the current ones, so that a load is in
    // flight during every encode (the loop is otherwise bound by the load latency)
    if (XT == SYN_Q8_0) {
        const int e = (lane & 7) * 4;
        auto load = [&](int64_t b) {
            return b < n_rows_blocks ? *reinterpret_cast<const float4*>(X + b * 32 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        };
        float4 xn = load(warp * 4 + (lane >> 3));
        for (int64_t base = warp * 4; base < n_rows_blocks; base += n_warps * 4) {
            const int64_t b = base + (lane >> 3);
            const float4 x = xn;
            xn = load(b + n_warps * 4);
            float v[4] = {x.x, x.y, x.z, x.w};
            float q[4];
            const uint16_t db = q8_0_group_codes(v, q);
            if (b < n_rows_blocks) {
                const float D = h2f_bits(db);
                __half2 a = __floats2half2_rn(__fmul_rn(D, q[0]), __fmul_rn(D, q[1]));
                __half2 c = __floats2half2_rn(__fmul_rn(D, q[2]), __fmul_rn(D, q[3]));
                uint2 out = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&c));
                *reinterpret_cast<uint2*>(xh + b * 32 + e) = out;
            }
        }
    } else {
        float4 n0 = make_float4(0.f, 0.f, 0.f, 0.f), n1 = n0;
        if (warp < n_rows_blocks) {
            n0 = *reinterpret_cast<const float4*>(X + warp * 256 + lane * 8);
            n1 = *reinterpret_cast<const float4*>(X + warp * 256 + lane * 8 + 4);
        }
        for (int64_t b = warp; b < n_rows_blocks; b += n_warps) {
            const float4 x0 = n0, x1 = n1;
            const int64_t bn = b + n_warps;
            if (bn < n_rows_blocks) {
                n0 = *reinterpret_cast<const float4*>(X + bn * 256 + lane * 8);
                n1 = *reinterpret_cast<const float4*>(X + bn * 256 + lane * 8 + 4);
            }
            float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            float q[8];
            const float dd = q8_k_warp_codes(v, q);
            uint32_t hv[4];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                __half2 h2 = __floats2half2_rn(__fmul_rn(dd, q[2 * k]), __fmul_rn(dd, q[2 * k + 1]));
                hv[k] = *reinterpret_cast<uint32_t*>(&h2);
            }
            if (SYN_IN_BOUNDS(b < n_rows_blocks))
                *reinterpret_cast<uint4*>(xh + b * 256 + lane * 8) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        }
    }
}

// ---------------------------------------------------------------------------------------
// integer block sums (bit-exact check of the block dot; not on the hot path)
// ---------------------------------------------------------------------------------------

template <int T>
__global__ void k_block_sums(const uint8_t* __restrict__ W, int64_t n_out, int64_t nb,
                             const uint8_t* __restrict__ Xq, int64_t n_tok,
                             int32_t* __restrict__ S) {
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t total = n_tok * n_out * nb;
    if (idx >= total) return;
    int64_t b = idx % nb;
    int64_t o = (idx / nb) % n_out;
    int64_t t = idx / (nb * n_out);
    int32_t s0 = 0, s1 = 0;
    if (T == SYN_Q4_0 || T == SYN_Q5_0) {
        constexpr int OFF = T == SYN_Q4_0 ? 8 : 16, BB = T == SYN_Q4_0 ? 18 : 22, QS = T == SYN_Q4_0 ? 2 : 6;
        const uint8_t* w = W + (o * nb + b) * BB;
        const uint8_t* x = Xq + (t * nb + b) * 34;
        const uint32_t qh = T == SYN_Q5_0 ? ((uint32_t)w[2] | ((uint32_t)w[3] << 8) | ((uint32_t)w[4] << 16) |
                                             ((uint32_t)w[5] << 24))
                                          : 0u;
        for (int i = 0; i < 32; i++) {
            int q = (w[QS + (i & 15)] >> (i >= 16 ? 4 : 0)) & 15;
            if (T == SYN_Q5_0) q |= (int)((qh >> i) & 1) << 4;
            s0 += (q - OFF) * (int32_t)(int8_t)x[2 + i];
        }
    } else if (T == SYN_Q8_0) {
        const uint8_t* w = W + (o * nb + b) * 34;
        const uint8_t* x = Xq + (t * nb + b) * 34;
        for (int i = 0; i < 32; i++) s0 += (int32_t)(int8_t)w[2 + i] * (int32_t)(int8_t)x[2 + i];
    } else {
        const uint8_t* x = Xq + (t * nb + b) * 292;
        const int8_t* xq = reinterpret_cast<const int8_t*>(x + 4);
        const int16_t* bs = reinterpret_cast<const int16_t*>(x + 260);
        if (T == SYN_Q4_K) {
            const uint8_t* w = W + (o * nb + b) * 144;
            const uint8_t* sb = w + 4;
            for (int j = 0; j < 8; j++) {
                int sc, mn;
                if (j < 4) { sc = sb[j] & 63; mn = sb[j + 4] & 63; }
                else { sc = (sb[j + 4] & 15) | ((sb[j - 4] >> 6) << 4); mn = (sb[j + 4] >> 4) | ((sb[j] >> 6) << 4); }
                int dot = 0;
                for (int l = 0; l < 32; l++) {
                    int q = (w[16 + 32 * (j >> 1) + l] >> ((j & 1) * 4)) & 15;
                    dot += q * xq[32 * j + l];
                }
                s0 += sc * dot;
                s1 += mn * (bs[2 * j] + bs[2 * j + 1]);
            }
        } else {
            const uint8_t* w = W + (o * nb + b) * 210;
            for (int i = 0; i < 256; i++) {
                int h = i >> 7, wi = i & 127, quarter = wi >> 5, l = wi & 31;
                int lo = (w[64 * h + l + ((quarter & 1) ? 32 : 0)] >> ((quarter >= 2) ? 4 : 0)) & 15;
                int hi = (w[128 + 32 * h + l] >> (2 * quarter)) & 3;
                int q = lo | (hi << 4);
                s0 += (int32_t)(int8_t)w[192 + (i >> 4)] * (q - 32) * xq[i];
            }
        }
    }
    S[idx * 2] = s0;
    S[idx * 2 + 1] = s1;
}

// ---------------------------------------------------------------------------------------
// F16 weights: the IEEE half of each value (round to nearest even); non-finite input or an
// overflow to infinity sets the range flag
// ---------------------------------------------------------------------------------------

__global__ void __launch_bounds__(256) k_quantize_f16(const float* __restrict__ src, __half* __restrict__ dst,
                                                      int64_t n, int* __restrict__ range_err) {
    bool ok = true;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float x = src[i];
        const __half h = __float2half_rn(x);
        ok &= isfinite(x) && !__hisinf(h);
        dst[i] = h;
    }
    if (!__all_sync(0xffffffffu, ok) && (threadIdx.x & 31) == 0) atomicExch(range_err, 1);
}

__global__ void __launch_bounds__(256) k_dequantize_f16(const __half* __restrict__ src, float* __restrict__ dst,
                                                        int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = __half2float(src[i]);
}

// ---------------------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------------------

static int grid_for(int64_t warps_needed, int sms) {
    int64_t ctas = (warps_needed + 7) / 8;
    int64_t cap = (int64_t)sms * 8;
    if (ctas > cap) ctas = cap;
    return ctas < 1 ? 1 : (int)ctas;
}

cudaError_t launch_quantize(int type, const float* src, void* dst, int64_t n_blocks, int* range_err,
                            int sms, cudaStream_t s) {
    if (type == SYN_F16) {
        k_quantize_f16<<<grid_for((n_blocks + 31) / 32, sms), 256, 0, s>>>(src, static_cast<__half*>(dst), n_blocks,
                                                                          range_err);
        return cudaGetLastError();
    }
    int64_t warps = small_block(type) ? (n_blocks + 3) / 4 : n_blocks;
    int g = grid_for(warps, sms);
    uint8_t* d = static_cast<uint8_t*>(dst);
    switch (type) {
    case SYN_Q8_0: k_quantize<SYN_Q8_0><<<g, 256, 0, s>>>(src, d, n_blocks, range_err); break;
    case SYN_Q4_K: k_quantize<SYN_Q4_K><<<g, 256, 0, s>>>(src, d, n_blocks, range_err); break;
    case SYN_Q6_K: k_quantize<SYN_Q6_K><<<g, 256, 0, s>>>(src, d, n_blocks, range_err); break;
    case SYN_Q8_K: k_quantize<SYN_Q8_K><<<g, 256, 0, s>>>(src, d, n_blocks, range_err); break;
    case SYN_Q4_0: k_quantize<SYN_Q4_0><<<g, 256, 0, s>>>(src, d, n_blocks, range_err); break;
    case SYN_Q5_0: k_quantize<SYN_Q5_0><<<g, 256, 0, s>>>(src, d, n_blocks, range_err); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_dequantize(int type, const void* src, float* dst, int64_t n_blocks, int sms,
                              cudaStream_t s) {
    if (type == SYN_F16) {
        k_dequantize_f16<<<grid_for((n_blocks + 31) / 32, sms), 256, 0, s>>>(static_cast<const __half*>(src), dst,
                                                                            n_blocks);
        return cudaGetLastError();
    }
    int64_t warps = small_block(type) ? (n_blocks + 3) / 4 : n_blocks;
    int g = grid_for(warps, sms);
    const uint8_t* p = static_cast<const uint8_t*>(src);
    switch (type) {
    case SYN_Q8_0: k_dequantize<SYN_Q8_0><<<g, 256, 0, s>>>(p, dst, n_blocks); break;
    case SYN_Q4_K: k_dequantize<SYN_Q4_K><<<g, 256, 0, s>>>(p, dst, n_blocks); break;
    case SYN_Q6_K: k_dequantize<SYN_Q6_K><<<g, 256, 0, s>>>(p, dst, n_blocks); break;
    case SYN_Q8_K: k_dequantize<SYN_Q8_K><<<g, 256, 0, s>>>(p, dst, n_blocks); break;
    case SYN_Q4_0: k_dequantize<SYN_Q4_0><<<g, 256, 0, s>>>(p, dst, n_blocks); break;
    case SYN_Q5_0: k_dequantize<SYN_Q5_0><<<g, 256, 0, s>>>(p, dst, n_blocks); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_deq_half(int type, const void* src, void* dst, int64_t n_blocks, int sms, cudaStream_t s) {
    // one wave of CTAs: as many per SM as are resident at once (the grid-stride loop does the
    // rest; a second, partial wave would leave SMs idle at its end)
    static std::atomic<int> per_sm_cache[2];  // 0: not known yet
    const int which = type == SYN_Q4_K ? 0 : 1;
    int per_sm = per_sm_cache[which].load();
    if (per_sm == 0) {
        int n = 0;
        const cudaError_t e = which == 0
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_deq_half<SYN_Q4_K>, 256, 0)
            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_deq_half<SYN_Q6_K>, 256, 0);
        per_sm = (e == cudaSuccess && n > 0) ? n : 4;
        per_sm_cache[which].store(per_sm);
    }
    int64_t ctas = ((n_blocks + DEQ_U - 1) / DEQ_U + 7) / 8;
    if (ctas > (int64_t)sms * per_sm) ctas = (int64_t)sms * per_sm;
    const int g = ctas < 1 ? 1 : (int)ctas;
    const uint8_t* p = static_cast<const uint8_t*>(src);
    __half* h = static_cast<__half*>(dst);
    switch (type) {
    case SYN_Q4_K: k_deq_half<SYN_Q4_K><<<g, 256, 0, s>>>(p, h, n_blocks); break;
    case SYN_Q6_K: k_deq_half<SYN_Q6_K><<<g, 256, 0, s>>>(p, h, n_blocks); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_quantize_act(int xtype, const float* X, int64_t n_blocks, int8_t* qs, float* d,
                                int16_t* bsums, int sms, cudaStream_t s) {
    int64_t warps = (xtype == SYN_Q8_0) ? (n_blocks + 3) / 4 : n_blocks;
    int g = grid_for(warps, sms);
    if (xtype == SYN_Q8_0) k_quantize_act<SYN_Q8_0><<<g, 256, 0, s>>>(X, n_blocks, qs, d, bsums);
    else k_quantize_act<SYN_Q8_K><<<g, 256, 0, s>>>(X, n_blocks, qs, d, bsums);
    return cudaGetLastError();
}

cudaError_t launch_act_half(int xtype, const float* X, int64_t n_blocks, void* xh, int sms,
                            cudaStream_t s) {
    if (xtype == SYN_F16) return launch_x_to_half(X, n_blocks, xh, sms, s);  // F16: rounding only
    const int64_t warps = (xtype == SYN_Q8_0) ? (n_blocks + 3) / 4 : n_blocks;
    // one wave of CTAs: as many per SM as are resident at once (the grid-stride loop does the
    // rest; a second, partial wave would leave SMs idle at its end)
    static std::atomic<int> per_sm_cache[2];  // 0: not known yet
    const int which = xtype == SYN_Q8_0 ? 0 : 1;
    int per_sm = per_sm_cache[which].load();
    if (per_sm == 0) {
        int n = 0;
        const cudaError_t e = which == 0
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_act_half<SYN_Q8_0>, 256, 0)
            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_act_half<SYN_Q8_K>, 256, 0);
        per_sm = (e == cudaSuccess && n > 0) ? n : 4;
        per_sm_cache[which].store(per_sm);
    }
    int64_t ctas = (warps + 7) / 8;
    if (ctas > (int64_t)sms * per_sm) ctas = (int64_t)sms * per_sm;
    const int g = ctas < 1 ? 1 : (int)ctas;
    __half* h = static_cast<__half*>(xh);
    if (xtype == SYN_Q8_0) k_act_half<SYN_Q8_0><<<g, 256, 0, s>>>(X, n_blocks, h);
    else k_act_half<SYN_Q8_K><<<g, 256, 0, s>>>(X, n_blocks, h);
    return cudaGetLastError();
}

cudaError_t launch_block_sums(int type, const void* W, int64_t n_out, int64_t nb, const void* Xq,
                              int64_t n_tok, int32_t* S, cudaStream_t s) {
    int64_t total = n_tok * n_out * nb;
    if (total == 0) return cudaSuccess;
    int64_t g = (total + 255) / 256;
    const uint8_t* w = static_cast<const uint8_t*>(W);
    const uint8_t* x = static_cast<const uint8_t*>(Xq);
    switch (type) {
    case SYN_Q8_0: k_block_sums<SYN_Q8_0><<<(unsigned)g, 256, 0, s>>>(w, n_out, nb, x, n_tok, S); break;
    case SYN_Q4_K: k_block_sums<SYN_Q4_K><<<(unsigned)g, 256, 0, s>>>(w, n_out, nb, x, n_tok, S); break;
    case SYN_Q6_K: k_block_sums<SYN_Q6_K><<<(unsigned)g, 256, 0, s>>>(w, n_out, nb, x, n_tok, S); break;
    case SYN_Q4_0: k_block_sums<SYN_Q4_0><<<(unsigned)g, 256, 0, s>>>(w, n_out, nb, x, n_tok, S); break;
    case SYN_Q5_0: k_block_sums<SYN_Q5_0><<<(unsigned)g, 256, 0, s>>>(w, n_out, nb, x, n_tok, S); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

#ifdef SYN_DEBUG
SYN_BOUNDS_READER(debug_bounds_quant)

// One check given an out-of-range index on purpose: idx = 4 against 4 checked elements.
// The guarded store is skipped; were the check ever compiled wrong, it would still land in
// the shared array (8 elements), never outside it.
__global__ void k_bounds_selftest(int n_checked) {
    __shared__ int slot[8];
    const int idx = n_checked;
    if (SYN_IN_BOUNDS(idx < n_checked)) slot[idx & 7] = 1;
}

cudaError_t launch_bounds_selftest(cudaStream_t s) {
    k_bounds_selftest<<<1, 32, 0, s>>>(4);
    return cudaGetLastError();
}
#endif

}  // namespace syn

// gemv.cu — decode product (few tokens): Y[t][o] = sum_b blockdot(W[o,b], Xq[t,b]).
//
// "The GGML ecosystem, and where synapse fits", section 5, "Products: weights against
// quantized activations": the activations are converted once per row to the weight
// format's vec_dot_type, each weight block is dotted with the matching activation block
// in integer arithmetic and only the per-block scales are float.  Decode streams every
// weight once per token group, so the kernel is bound by HBM bandwidth ("llama.cpp and
// GGUF", CPU and Edge Inference: tokens/s <= bandwidth / model size).
//
// One launch does everything:
//   1. each CTA quantizes the (<= NT) activation rows into shared memory with the same
//      encoder as syn_quantize_activations (codes, scales, 16-sums);
//   2. each warp streams its own weight rows, R rows at a time, through an NS-deep ring of
//      shared-memory stages filled by 1-D bulk copies (cp.async.bulk, completion on an
//      mbarrier).  The copy window is widened to 16-byte boundaries, so the 34- and
//      210-byte blocks need no alignment;
//   3. lanes unpack 4/6/8-bit codes in registers, form the integer block dots with dp4a,
//      apply the fp32 block scales and keep R x NT partial sums; a warp reduction ends each
//      row group.
#include <algorithm>

#include "kernels.h"
#include "quant_dev.cuh"

namespace syn {

struct GemvParams {
    const uint8_t* W;
    const float* X;
    float* Y;
    int* err;
    int64_t n_out, n_in, n_tok;
    int64_t row_bytes;
    int64_t total_floor16;  // W byte count rounded down to 16
    int64_t n_groups;       // ceil(n_out / R)
    int nb;                 // blocks per row
    int cb;                 // blocks per chunk
    int n_chunks;           // chunks per row
    int slot;               // bytes per row slot of a stage
    int nbx;                // activation blocks per row
    int off_d, off_bs, off_stage, off_bar, off_flag;
};

template <int T> struct GemvFmt;
template <> struct GemvFmt<SYN_Q4_K> { static constexpr int U = 4, BB = 144, XT = SYN_Q8_K, BX = 256; };
template <> struct GemvFmt<SYN_Q6_K> { static constexpr int U = 4, BB = 210, XT = SYN_Q8_K, BX = 256; };
template <> struct GemvFmt<SYN_Q8_0> { static constexpr int U = 16, BB = 34, XT = SYN_Q8_0, BX = 32; };

constexpr int GEMV_WARPS = 8;

// Four 32-bit words starting at any even shared-memory address.
__device__ __forceinline__ void lds_u32x4_any(const uint8_t* p, uint32_t out[4]) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    uint32_t sh = static_cast<uint32_t>(a & 3) * 8;
    uint32_t v[5];
#pragma unroll
    for (int i = 0; i < 5; i++) v[i] = w[i];
#pragma unroll
    for (int i = 0; i < 4; i++) out[i] = __funnelshift_r(v[i], v[i + 1], sh);
}

__device__ __forceinline__ void lds_u32x2_any(const uint8_t* p, uint32_t out[2]) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    uint32_t sh = static_cast<uint32_t>(a & 3) * 8;
    uint32_t v0 = w[0], v1 = w[1], v2 = w[2];
    out[0] = __funnelshift_r(v0, v1, sh);
    out[1] = __funnelshift_r(v1, v2, sh);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Quantize activation rows t0 .. t0+NT-1 (rows >= n_tok become zeros) into shared memory.
template <int XT, int NT>
__device__ void act_to_smem(const GemvParams& p, int64_t t0, uint8_t* smem) {
    int8_t* aq = reinterpret_cast<int8_t*>(smem);
    float* ad = reinterpret_cast<float*>(smem + p.off_d);
    int16_t* abs_ = reinterpret_cast<int16_t*>(smem + p.off_bs);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nbx = p.nbx;
    if (XT == SYN_Q8_0) {
        const int steps = (nbx + 3) / 4;  // 4 blocks per warp step
        for (int k = warp; k < NT * steps; k += GEMV_WARPS) {
            int t = k / steps, b = (k % steps) * 4 + (lane >> 3), e = (lane & 7) * 4;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            bool live = (t0 + t < p.n_tok) && (b < nbx);
            if (live) {
                float4 x = *reinterpret_cast<const float4*>(p.X + (t0 + t) * p.n_in + b * 32 + e);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            }
            uint16_t db;
            bool fin;
            uint32_t q = q8_0_group(v, &db, &fin);
            if (b < nbx) {
                *reinterpret_cast<uint32_t*>(aq + t * p.n_in + b * 32 + e) = q;
                if ((lane & 7) == 0) ad[t * nbx + b] = h2f_bits(db);
            }
        }
    } else {
        for (int k = warp; k < NT * nbx; k += GEMV_WARPS) {
            int t = k / nbx, b = k % nbx;
            float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (t0 + t < p.n_tok) {
                const float* x = p.X + (t0 + t) * p.n_in + b * 256 + lane * 8;
                float4 x0 = *reinterpret_cast<const float4*>(x);
                float4 x1 = *reinterpret_cast<const float4*>(x + 4);
                v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
                v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
            }
            uint32_t w0, w1;
            float dd;
            int bs;
            bool fin;
            q8_k_warp(v, &w0, &w1, &dd, &bs, &fin);
            *reinterpret_cast<uint2*>(aq + t * p.n_in + b * 256 + lane * 8) = make_uint2(w0, w1);
            if (lane == 0) ad[t * nbx + b] = dd;
            if ((lane & 1) == 0) abs_[(t * nbx + b) * 16 + (lane >> 1)] = (int16_t)bs;
        }
    }
}

template <int T, int NT, int R, int NS>
__global__ void __launch_bounds__(GEMV_WARPS * 32) k_gemv(const GemvParams p) {
    using F = GemvFmt<T>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * GEMV_WARPS + warp;
    const int64_t GW = (int64_t)gridDim.x * GEMV_WARPS;
    uint8_t* stages = smem + p.off_stage + (size_t)warp * NS * R * p.slot;
    const uint32_t stage_addr = smem_u32(stages);
    const uint32_t bar0 = smem_u32(smem + p.off_bar) + warp * NS * 8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.off_flag);

    if (threadIdx.x == 0) *abort_flag = 0;
    if (lane == 0)
        for (int s = 0; s < NS; s++) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
    __syncthreads();

    const int8_t* aq = reinterpret_cast<const int8_t*>(smem);
    const float* ad = reinterpret_cast<const float*>(smem + p.off_d);
    const int16_t* abs_ = reinterpret_cast<const int16_t*>(smem + p.off_bs);

    const int64_t my_groups = gw < p.n_groups ? (p.n_groups - 1 - gw) / GW + 1 : 0;
    const int64_t n_tasks = my_groups * p.n_chunks;
    uint32_t seq = 0;  // running stage-use counter of this warp (all token chunks)

    // Issue the bulk copies of task i (group, chunk) into stage seq_i % NS.
    auto issue = [&](int64_t i, uint32_t seq_i) {
        const int64_t g = gw + (i / p.n_chunks) * GW;
        const int c = (int)(i % p.n_chunks);
        const int nblk = min(p.cb, p.nb - c * p.cb);
        const int s = seq_i % NS;
        const uint32_t bar = bar0 + 8 * s;
        uint8_t* sbase = stages + (size_t)s * R * p.slot;
        __syncwarp();
        if (lane == 0) {
            fence_proxy_async_smem();
            uint32_t tx = 0;
            int64_t a0s[R], bytes[R];
#pragma unroll
            for (int r = 0; r < R; r++) {
                a0s[r] = 0; bytes[r] = 0;
                const int64_t o = g * R + r;
                if (o >= p.n_out) continue;
                const int64_t src = o * p.row_bytes + (int64_t)c * p.cb * F::BB;
                const int64_t a0 = src & ~int64_t(15);
                int64_t a1 = (src + (int64_t)nblk * F::BB + 15) & ~int64_t(15);
                if (a1 > p.total_floor16) a1 = p.total_floor16;
                a0s[r] = a0;
                bytes[r] = a1 > a0 ? a1 - a0 : 0;
                tx += (uint32_t)bytes[r];
            }
            mbar_arrive_expect_tx(bar, tx);
#pragma unroll
            for (int r = 0; r < R; r++)
                if (bytes[r] > 0)
                    bulk_g2s(stage_addr + (uint32_t)((s * R + r) * p.slot), p.W + a0s[r],
                             (uint32_t)bytes[r], bar);
        }
        // The last (< 16) bytes of W, past the last 16-byte boundary, by plain loads.
#pragma unroll
        for (int r = 0; r < R; r++) {
            const int64_t o = g * R + r;
            if (o >= p.n_out) continue;
            const int64_t src = o * p.row_bytes + (int64_t)c * p.cb * F::BB;
            const int64_t end = src + (int64_t)nblk * F::BB;
            if (end > p.total_floor16) {
                const int64_t a0 = src & ~int64_t(15);
                const int64_t from = p.total_floor16 > a0 ? p.total_floor16 : a0;
                const int64_t k = from + lane;
                if (k < end) sbase[r * p.slot + (k - a0)] = p.W[k];
            }
        }
        __syncwarp();
    };

    for (int64_t t0 = 0; t0 < p.n_tok; t0 += NT) {
        __syncthreads();  // every warp is done with the previous token chunk
        act_to_smem<F::XT, NT>(p, t0, smem);
        __syncthreads();
        if (*abort_flag) break;

        const int npre = (int)(n_tasks < NS - 1 ? n_tasks : NS - 1);
        for (int i = 0; i < npre; i++) issue(i, seq + i);

        float acc[R][NT];
        for (int64_t i = 0; i < n_tasks; i++) {
            if (i + NS - 1 < n_tasks) issue(i + NS - 1, seq + (uint32_t)(i + NS - 1));
            const uint32_t q = seq + (uint32_t)i;
            const int s = q % NS;
            if (!mbar_wait(bar0 + 8 * s, (q / NS) & 1, p.err, abort_flag)) {
                // Drain the copies this warp still has in flight (bounded), so that no
                // bulk copy targets the shared memory of a finished CTA.
                const int64_t hi = (n_tasks < i + NS - 1) ? n_tasks : i + NS - 1;
                for (int64_t k = i; k < hi; k++) {
                    const uint32_t qk = seq + (uint32_t)k;
                    long long w0 = clock64();
                    while (!mbar_try_wait(bar0 + 8 * (qk % NS), (qk / NS) & 1) &&
                           clock64() - w0 < SYN_WAIT_CYCLES / 8) {
                    }
                }
                break;
            }

            const int64_t g = gw + (i / p.n_chunks) * GW;
            const int c = (int)(i % p.n_chunks);
            const int nblk = min(p.cb, p.nb - c * p.cb);
            if (c == 0) {
#pragma unroll
                for (int r = 0; r < R; r++)
#pragma unroll
                    for (int t = 0; t < NT; t++) acc[r][t] = 0.f;
            }
            const uint8_t* sbase = stages + (size_t)s * R * p.slot;
            int delta[R];
#pragma unroll
            for (int r = 0; r < R; r++)
                delta[r] = (int)(((g * R + r) * p.row_bytes + (int64_t)c * p.cb * F::BB) & 15);

            for (int u = 0; u * F::U < nblk; u++) {
                if (T == SYN_Q4_K) {
                    const int kb = u * 4 + (lane >> 3);
                    if (kb < nblk) {
                        const int part = lane & 7, cc = part >> 1, hlf = part & 1;
                        const int B = c * p.cb + kb;
                        uint4 xlo[NT], xhi[NT];
                        float dx[NT];
                        int xs_lo[NT], xs_hi[NT];
#pragma unroll
                        for (int t = 0; t < NT; t++) {
                            const int8_t* xq = aq + t * p.n_in + B * 256 + 64 * cc + 16 * hlf;
                            xlo[t] = *reinterpret_cast<const uint4*>(xq);
                            xhi[t] = *reinterpret_cast<const uint4*>(xq + 32);
                            dx[t] = ad[t * p.nbx + B];
                            const int16_t* bs = abs_ + (t * p.nbx + B) * 16 + 4 * cc;
                            xs_lo[t] = hlf ? 0 : (int)bs[0] + (int)bs[1];
                            xs_hi[t] = hlf ? 0 : (int)bs[2] + (int)bs[3];
                        }
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            const uint8_t* blk = sbase + r * p.slot + delta[r] + kb * 144;
                            const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
                            const uint4 qv = *reinterpret_cast<const uint4*>(blk + 16 + 32 * cc + 16 * hlf);
                            const float D = h2f_bits(hdr.x & 0xFFFF), Dm = h2f_bits(hdr.x >> 16);
                            // scales/mins of sub-blocks j = 2cc (low nibbles) and 2cc+1 (high)
                            int sc[2], mn[2];
#pragma unroll
                            for (int h = 0; h < 2; h++) {
                                const int j = 2 * cc + h, jj = j & 3, sh = 8 * jj;
                                const int lo_sc = (hdr.y >> sh) & 63, lo_mn = (hdr.z >> sh) & 63;
                                const int hi_sc = ((hdr.w >> sh) & 15) | (((hdr.y >> (sh + 6)) & 3) << 4);
                                const int hi_mn = ((hdr.w >> (sh + 4)) & 15) | (((hdr.z >> (sh + 6)) & 3) << 4);
                                sc[h] = j < 4 ? lo_sc : hi_sc;
                                mn[h] = j < 4 ? lo_mn : hi_mn;
                            }
                            const uint32_t l0 = qv.x & 0x0F0F0F0Fu, l1 = qv.y & 0x0F0F0F0Fu;
                            const uint32_t l2 = qv.z & 0x0F0F0F0Fu, l3 = qv.w & 0x0F0F0F0Fu;
                            const uint32_t h0 = (qv.x >> 4) & 0x0F0F0F0Fu, h1 = (qv.y >> 4) & 0x0F0F0F0Fu;
                            const uint32_t h2 = (qv.z >> 4) & 0x0F0F0F0Fu, h3 = (qv.w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                            for (int t = 0; t < NT; t++) {
                                int dl = dp4a(l0, xlo[t].x, 0);
                                dl = dp4a(l1, xlo[t].y, dl);
                                dl = dp4a(l2, xlo[t].z, dl);
                                dl = dp4a(l3, xlo[t].w, dl);
                                int dh = dp4a(h0, xhi[t].x, 0);
                                dh = dp4a(h1, xhi[t].y, dh);
                                dh = dp4a(h2, xhi[t].z, dh);
                                dh = dp4a(h3, xhi[t].w, dh);
                                const int A = sc[0] * dl + sc[1] * dh;
                                const int Bm = mn[0] * xs_lo[t] + mn[1] * xs_hi[t];
                                acc[r][t] = fmaf(dx[t], D * (float)A - Dm * (float)Bm, acc[r][t]);
                            }
                        }
                    }
                } else if (T == SYN_Q6_K) {
                    const int kb = u * 4 + (lane >> 3);
                    if (kb < nblk) {
                        const int part = lane & 7, H = part >> 2, l0 = 8 * (part & 3);
                        const bool corr = (l0 & 15) == 0;
                        const int B = c * p.cb + kb;
                        uint2 xw[NT][4];
                        float dx[NT];
                        int bsk[NT][4];
#pragma unroll
                        for (int t = 0; t < NT; t++) {
                            const int8_t* xq = aq + t * p.n_in + B * 256 + 128 * H + l0;
#pragma unroll
                            for (int k = 0; k < 4; k++) xw[t][k] = *reinterpret_cast<const uint2*>(xq + 32 * k);
                            dx[t] = ad[t * p.nbx + B];
                            const int16_t* bs = abs_ + (t * p.nbx + B) * 16 + 8 * H + (l0 >> 4);
#pragma unroll
                            for (int k = 0; k < 4; k++) bsk[t][k] = corr ? (int)bs[2 * k] : 0;
                        }
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            const uint8_t* blk = sbase + r * p.slot + delta[r] + kb * 210;
                            uint32_t qa[2], qb[2], qh[2];
                            lds_u32x2_any(blk + 64 * H + l0, qa);
                            lds_u32x2_any(blk + 64 * H + 32 + l0, qb);
                            lds_u32x2_any(blk + 128 + 32 * H + l0, qh);
                            int sc[4];
#pragma unroll
                            for (int k = 0; k < 4; k++)
                                sc[k] = (int)reinterpret_cast<const int8_t*>(blk)[192 + 8 * H + 2 * k + (l0 >> 4)];
                            const float D = h2f_bits(*reinterpret_cast<const uint16_t*>(blk + 208));
                            uint32_t q[4][2];
#pragma unroll
                            for (int w = 0; w < 2; w++) {
                                q[0][w] = (qa[w] & 0x0F0F0F0Fu) | ((qh[w] << 4) & 0x30303030u);
                                q[1][w] = (qb[w] & 0x0F0F0F0Fu) | ((qh[w] << 2) & 0x30303030u);
                                q[2][w] = ((qa[w] >> 4) & 0x0F0F0F0Fu) | (qh[w] & 0x30303030u);
                                q[3][w] = ((qb[w] >> 4) & 0x0F0F0F0Fu) | ((qh[w] >> 2) & 0x30303030u);
                            }
#pragma unroll
                            for (int t = 0; t < NT; t++) {
                                int C = 0, cs = 0;
#pragma unroll
                                for (int k = 0; k < 4; k++) {
                                    int dk = dp4a(q[k][0], xw[t][k].x, 0);
                                    dk = dp4a(q[k][1], xw[t][k].y, dk);
                                    C += sc[k] * dk;
                                    cs += sc[k] * bsk[t][k];
                                }
                                C -= 32 * cs;
                                acc[r][t] = fmaf(dx[t] * D, (float)C, acc[r][t]);
                            }
                        }
                    }
                } else {  // Q8_0
                    const int kb = u * 16 + (lane >> 1);
                    if (kb < nblk) {
                        const int hlf = lane & 1;
                        const int B = c * p.cb + kb;
                        uint4 xw[NT];
                        float dx[NT];
#pragma unroll
                        for (int t = 0; t < NT; t++) {
                            xw[t] = *reinterpret_cast<const uint4*>(aq + t * p.n_in + B * 32 + 16 * hlf);
                            dx[t] = ad[t * p.nbx + B];
                        }
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            const uint8_t* blk = sbase + r * p.slot + delta[r] + kb * 34;
                            const float Dw = h2f_bits(*reinterpret_cast<const uint16_t*>(blk));
                            uint32_t w[4];
                            lds_u32x4_any(blk + 2 + 16 * hlf, w);
#pragma unroll
                            for (int t = 0; t < NT; t++) {
                                int I = dp4a(w[0], xw[t].x, 0);
                                I = dp4a(w[1], xw[t].y, I);
                                I = dp4a(w[2], xw[t].z, I);
                                I = dp4a(w[3], xw[t].w, I);
                                acc[r][t] = fmaf(Dw * dx[t], (float)I, acc[r][t]);
                            }
                        }
                    }
                }
            }

            if (c == p.n_chunks - 1) {
#pragma unroll
                for (int r = 0; r < R; r++) {
                    const int64_t o = g * R + r;
#pragma unroll
                    for (int t = 0; t < NT; t++) {
                        const float v = warp_sum(acc[r][t]);
                        if (lane == 0 && o < p.n_out && t0 + t < p.n_tok) p.Y[(t0 + t) * p.n_out + o] = v;
                    }
                }
            }
        }
        seq += (uint32_t)n_tasks;
    }
}

// ---------------------------------------------------------------------------------------
// host side: geometry, shared-memory layout, launch
// ---------------------------------------------------------------------------------------

static int64_t up16(int64_t v) { return (v + 15) & ~int64_t(15); }

template <int T, int NT, int R, int NS>
static cudaError_t run_gemv(GemvParams p, int sms, cudaStream_t s) {
    using F = GemvFmt<T>;
    // rows per stage slot: a chunk of cb blocks; keep a warp's ring near 12 KB
    const int slot_target = 12 * 1024 / (NS * R);
    int cb = std::max(1, (slot_target - 32) / F::BB / F::U) * F::U;
    if (cb > p.nb) cb = ((p.nb + F::U - 1) / F::U) * F::U;
    p.cb = cb;
    p.n_chunks = (p.nb + cb - 1) / cb;
    p.slot = (int)up16((int64_t)cb * F::BB + 32);
    p.nbx = (int)(p.n_in / F::BX);
    const int64_t act_q = up16((int64_t)NT * p.n_in);
    const int64_t act_d = up16((int64_t)NT * p.nbx * 4);
    const int64_t act_b = F::XT == SYN_Q8_K ? up16((int64_t)NT * (p.n_in / 16) * 2) : 16;
    p.off_d = (int)act_q;
    p.off_bs = (int)(act_q + act_d);
    int64_t off = act_q + act_d + act_b;
    off = (off + 127) & ~int64_t(127);
    p.off_stage = (int)off;
    off += (int64_t)GEMV_WARPS * NS * R * p.slot;
    p.off_bar = (int)off;
    off += GEMV_WARPS * NS * 8;
    p.off_flag = (int)off;
    off += 16;
    const size_t smem = (size_t)off;
    auto kern = k_gemv<T, NT, R, NS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, GEMV_WARPS * 32, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    p.n_groups = (p.n_out + R - 1) / R;
    int64_t ctas = (p.n_groups + GEMV_WARPS - 1) / GEMV_WARPS;
    ctas = std::min<int64_t>(ctas, (int64_t)sms * occ);
    kern<<<(unsigned)ctas, GEMV_WARPS * 32, smem, s>>>(p);
    return cudaGetLastError();
}

// Largest activation smem (bytes) the decode kernel uses per token chunk.
static constexpr int64_t GEMV_ACT_BUDGET = 72 * 1024;

template <int T>
static cudaError_t gemv_dispatch(GemvParams p, int sms, cudaStream_t s) {
    const int64_t per_tok = p.n_in + p.n_in / 8 + 16;  // codes + scales + sums (bound)
    int nt = 1;
    while (nt < 8 && nt < p.n_tok && (int64_t)(2 * nt) * per_tok <= GEMV_ACT_BUDGET) nt *= 2;
    if ((int64_t)nt * per_tok > GEMV_ACT_BUDGET && nt > 1) nt /= 2;
    switch (nt) {
    case 1: return run_gemv<T, 1, 2, 4>(p, sms, s);
    case 2: return run_gemv<T, 2, 2, 4>(p, sms, s);
    case 4: return run_gemv<T, 4, 4, 3>(p, sms, s);
    default: return run_gemv<T, 8, 2, 3>(p, sms, s);
    }
}

cudaError_t launch_gemv(int type, const void* W, int64_t n_out, int64_t n_in, const float* X,
                        int64_t n_tok, float* Y, int* err, int sms, cudaStream_t s) {
    GemvParams p{};
    p.W = static_cast<const uint8_t*>(W);
    p.X = X;
    p.Y = Y;
    p.err = err;
    p.n_out = n_out;
    p.n_in = n_in;
    p.n_tok = n_tok;
    p.nb = (int)(n_in / block_elems(type));
    p.row_bytes = (int64_t)p.nb * block_bytes(type);
    p.total_floor16 = (n_out * p.row_bytes) & ~int64_t(15);
    switch (type) {
    case SYN_Q8_0: return gemv_dispatch<SYN_Q8_0>(p, sms, s);
    case SYN_Q4_K: return gemv_dispatch<SYN_Q4_K>(p, sms, s);
    case SYN_Q6_K: return gemv_dispatch<SYN_Q6_K>(p, sms, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace syn

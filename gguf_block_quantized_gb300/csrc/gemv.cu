// gemv.cu — decode product (few tokens): Y[t][o] = sum_b blockdot(W[o,b], Xq[t,b]), for one
// weight matrix or for a group of independent matrices in a single launch.
//
// "The GGML ecosystem, and where synapse fits", section 5, "Products: weights against
// quantized activations": the activations are converted once per row to the weight
// format's vec_dot_type, each weight block is dotted with the matching activation block
// in integer arithmetic and only the per-block scales are float.  Decode streams every
// weight once per token group, so the kernel is bound by HBM bandwidth ("llama.cpp and
// GGUF", CPU and Edge Inference: tokens/s <= bandwidth / model size).
//
// One CTA per SM.  The weight bytes of all matrices of the launch, row after row, are cut
// at row boundaries into one contiguous range per warp of about equal size.
//   1. Each warp starts its 1-D bulk copies (cp.async.bulk, completion on an mbarrier)
//      into its own 3-deep ring of shared-memory stages: a stage is a run of whole blocks,
//      copied through a window widened to 16-byte boundaries (so 34- and 210-byte blocks
//      need no alignment); bytes past the last 16-byte boundary of W come by plain loads.
//   2. Meanwhile the CTA converts the activation rows of the matrices its warps touch into
//      shared memory, with the same encoder as syn_quantize_activations, in a swizzled
//      layout: the 16-byte chunks of consecutive blocks land in different bank groups.
//   3. Each lane decodes whole blocks (one per warp step): unpacks 4/6/8-bit codes in
//      registers, forms the integer sub-block dots with dp4a, applies the integer sub-block
//      scales and then the fp32 block scales.  Rows of at most 32 blocks are spread over
//      groups of lanes (several rows per step, reduced within the group); wider rows take
//      several steps and a whole-warp reduction.
#include <algorithm>
#include <mutex>

#include "kernels.h"
#include "quant_dev.cuh"

namespace syn {

// Launch geometry (compile-time; the defaults are the measured best on GB300).
#ifndef SYN_GV_WARPS
#define SYN_GV_WARPS 8
#endif
#ifndef SYN_GV_NS
#define SYN_GV_NS 3
#endif
#ifndef SYN_GV_STAGE
#define SYN_GV_STAGE 8192
#endif
constexpr int GV_WARPS = SYN_GV_WARPS;
constexpr int GV_NS = SYN_GV_NS;            // stages per warp ring
constexpr int GV_STAGE = SYN_GV_STAGE;      // bytes of whole blocks per stage (at most)
constexpr int GV_SLOT = GV_STAGE + 32;      // stage slot: data plus the alignment window
// A stage must hold one warp step (32 blocks) of the widest block (Q6_K, 210 bytes).
static_assert(GV_STAGE >= 32 * 210, "decode stage smaller than one warp step of blocks");

struct GemvJob {
    const uint8_t* W;
    const float* X;
    float* Y;
    int64_t n_out;
    int64_t row_bytes;
    int64_t total_floor16;  // W byte count rounded down to 16
    int64_t byte_begin;     // offset of this matrix in the concatenated weight bytes
    int n_in, type, nb, bb;
    int stage_blocks;       // blocks per stage
    int lg_nb;              // log2(nb) when rows are packed several per warp step, else -1
    int nbx;                // activation blocks per row
    int act_q, act_d, act_s;  // shared-memory offsets of the converted activations
};

struct GemvBatch {
    GemvJob job[GEMV_MAX_JOBS];
    int n_jobs;
    int64_t total_bytes;
    int64_t n_tok;
    int* err;
    int off_stage, off_bar, off_flag;
};

// N 32-bit words starting at any even shared-memory address (aligned loads, funnel shift).
template <int N>
__device__ __forceinline__ void lds_words_any(const uint8_t* p, uint32_t* out) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3) * 8;
    uint32_t prev = w[0];
#pragma unroll
    for (int i = 0; i < N; i++) {
        const uint32_t nxt = w[i + 1];
        out[i] = __funnelshift_r(prev, nxt, sh);
        prev = nxt;
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over aligned groups of 2^lg lanes (lg <= 5).
__device__ __forceinline__ float group_sum(float v, int lg) {
#pragma unroll
    for (int k = 0; k < 5; k++)
        if (k < lg) v += __shfl_xor_sync(0xffffffffu, v, 1 << k);
    return v;
}

// Swizzled activation chunks: byte offset of chunk c (16 bytes) of block B.
__device__ __forceinline__ int k_chunk(int B, int c) { return 256 * B + 16 * (c ^ (B & 7)); }
__device__ __forceinline__ int q8_chunk(int B, int c) { return 32 * B + 16 * (c ^ ((B >> 2) & 1)); }

// First row boundary at or after byte t of the concatenated weights: (job, row).
__device__ __forceinline__ void row_at(const GemvBatch& b, int64_t t, int& j, int64_t& r) {
    j = 0;
    while (j < b.n_jobs - 1 && t >= b.job[j + 1].byte_begin) j++;
    const GemvJob& J = b.job[j];
    const int64_t off = t - J.byte_begin;
    r = (off + J.row_bytes - 1) / J.row_bytes;
    if (r >= J.n_out && j < b.n_jobs - 1) {
        j++;
        r = 0;
    } else if (r > J.n_out) {
        r = J.n_out;
    }
}

// Convert activation rows t0 .. t0+NT-1 of jobs [ja, jb] into shared memory (swizzled).
template <int NT>
__device__ void act_to_smem(const GemvBatch& b, int ja, int jb, int64_t t0, uint8_t* smem) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int j = ja; j <= jb; j++) {
        const GemvJob& J = b.job[j];
        int8_t* aq = reinterpret_cast<int8_t*>(smem + J.act_q);
        float* ad = reinterpret_cast<float*>(smem + J.act_d);
        int16_t* as = reinterpret_cast<int16_t*>(smem + J.act_s);
        const int nbx = J.nbx;
        if (J.type == SYN_Q8_0) {
            const int steps = (nbx + 3) / 4;  // 4 blocks of 32 per warp step
            for (int k = warp; k < NT * steps; k += GV_WARPS) {
                const int t = k / steps, blk = (k % steps) * 4 + (lane >> 3), e = lane & 7;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (t0 + t < b.n_tok && blk < nbx) {
                    const float4 x = *reinterpret_cast<const float4*>(J.X + (t0 + t) * J.n_in + blk * 32 + 4 * e);
                    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
                }
                uint16_t db;
                bool fin;
                const uint32_t q = q8_0_group(v, &db, &fin);
                if (blk < nbx) {
                    *reinterpret_cast<uint32_t*>(aq + t * J.n_in + q8_chunk(blk, e >> 2) + 4 * (e & 3)) = q;
                    if (e == 0) ad[t * nbx + blk] = h2f_bits(db);
                }
            }
        } else {
            for (int k = warp; k < NT * nbx; k += GV_WARPS) {
                const int t = k / nbx, blk = k % nbx;
                float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (t0 + t < b.n_tok) {
                    const float* x = J.X + (t0 + t) * J.n_in + blk * 256 + lane * 8;
                    const float4 x0 = *reinterpret_cast<const float4*>(x);
                    const float4 x1 = *reinterpret_cast<const float4*>(x + 4);
                    v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
                    v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
                }
                uint32_t w0, w1;
                float dd;
                int bs;
                bool fin;
                q8_k_warp(v, &w0, &w1, &dd, &bs, &fin);
                *reinterpret_cast<uint2*>(aq + t * J.n_in + k_chunk(blk, lane >> 1) + 8 * (lane & 1)) =
                    make_uint2(w0, w1);
                if (lane == 0) ad[t * nbx + blk] = dd;
                if ((lane & 1) == 0) as[(t * nbx + blk) * 16 + (lane >> 1)] = (int16_t)bs;
            }
        }
    }
}

struct ActView {
    const int8_t* q;    // token 0 codes (swizzled chunks); token t at + t * n_in
    const float* d;     // token 0 scales; token t at + t * nbx
    const int16_t* s;   // token 0 16-sums; token t at + t * nbx * 16
    int n_in, nbx;
};

// ---- one whole block per lane: Q4_K (144 bytes, 16-byte aligned in shared memory) ----
template <int NT>
__device__ __forceinline__ void blk_q4_k(const uint8_t* blk, int B, const ActView& A, float acc[NT]) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const float D = h2f_bits(hdr.x & 0xFFFF), Dm = h2f_bits(hdr.x >> 16);
    int sc[8], mn[8];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        sc[j] = (hdr.y >> (8 * j)) & 63;
        mn[j] = (hdr.z >> (8 * j)) & 63;
        sc[j + 4] = ((hdr.w >> (8 * j)) & 15) | (((hdr.y >> (8 * j + 6)) & 3) << 4);
        mn[j + 4] = ((hdr.w >> (8 * j + 4)) & 15) | (((hdr.z >> (8 * j + 6)) & 3) << 4);
    }
    int At[NT];
#pragma unroll
    for (int t = 0; t < NT; t++) At[t] = 0;
#pragma unroll
    for (int c = 0; c < 4; c++) {  // 32 code bytes: sub-block 2c (low nibbles), 2c+1 (high)
        const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
        const uint32_t q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const int8_t* xq = A.q + t * A.n_in;
            const uint4 x0 = *reinterpret_cast<const uint4*>(xq + k_chunk(B, 4 * c));
            const uint4 x1 = *reinterpret_cast<const uint4*>(xq + k_chunk(B, 4 * c + 1));
            const uint4 x2 = *reinterpret_cast<const uint4*>(xq + k_chunk(B, 4 * c + 2));
            const uint4 x3 = *reinterpret_cast<const uint4*>(xq + k_chunk(B, 4 * c + 3));
            const uint32_t xl[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const uint32_t xh[8] = {x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
            int dl = 0, dh = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                dl = dp4a(q[i] & 0x0F0F0F0Fu, xl[i], dl);
                dh = dp4a((q[i] >> 4) & 0x0F0F0F0Fu, xh[i], dh);
            }
            At[t] += sc[2 * c] * dl + sc[2 * c + 1] * dh;
        }
    }
#pragma unroll
    for (int t = 0; t < NT; t++) {
        const uint4* sp = reinterpret_cast<const uint4*>(A.s + (t * A.nbx + B) * 16);
        const uint4 s0 = sp[0], s1 = sp[1];
        const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        int Bm = 0;
#pragma unroll
        for (int j = 0; j < 8; j++)  // sub-block j of 32 = 16-sums 2j, 2j+1 = halves of word j
            Bm += mn[j] * ((int)(int16_t)(sw[j] & 0xFFFF) + (int)(int16_t)(sw[j] >> 16));
        acc[t] = fmaf(A.d[t * A.nbx + B], D * (float)At[t] - Dm * (float)Bm, acc[t]);
    }
}

// ---- one whole block per lane: Q6_K (210 bytes, 2-byte aligned) ----
template <int NT>
__device__ __forceinline__ void blk_q6_k(const uint8_t* blk, int B, const ActView& A, float acc[NT]) {
    const float D = h2f_bits(*reinterpret_cast<const uint16_t*>(blk + 208));
    uint32_t scw[4];
    lds_words_any<4>(blk + 192, scw);
    int Ct[NT];
#pragma unroll
    for (int t = 0; t < NT; t++) Ct[t] = 0;
#pragma unroll
    for (int H = 0; H < 2; H++) {
        uint32_t ql[16], qh[8];
        lds_words_any<16>(blk + 64 * H, ql);
        lds_words_any<8>(blk + 128 + 32 * H, qh);
        // quarter k of the half, l = 4w..4w+3 (w = 4*half + i): sub-block 8H + 2k + half
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const int8_t* xq = A.q + t * A.n_in;
            int dot[8];
#pragma unroll
            for (int k = 0; k < 4; k++) {
#pragma unroll
                for (int half = 0; half < 2; half++) {
                    const uint4 x = *reinterpret_cast<const uint4*>(xq + k_chunk(B, 8 * H + 2 * k + half));
                    const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
                    int dsum = 0;
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int w = 4 * half + i;
                        const uint32_t a = (k & 1) ? ql[8 + w] : ql[w];
                        const uint32_t lo = (k >= 2) ? ((a >> 4) & 0x0F0F0F0Fu) : (a & 0x0F0F0F0Fu);
                        const uint32_t hi = (k >= 2 ? (qh[w] >> (2 * k - 4)) : (qh[w] << (4 - 2 * k))) & 0x30303030u;
                        dsum = dp4a(lo | hi, xw[i], dsum);
                    }
                    dot[2 * k + half] = dsum;
                }
            }
            const uint4 s = *reinterpret_cast<const uint4*>(A.s + (t * A.nbx + B) * 16 + 8 * H);
            const uint32_t sw[4] = {s.x, s.y, s.z, s.w};  // 16-sums of sub-blocks 8H .. 8H+7
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int bs = (int)(int16_t)((sw[j >> 1] >> (16 * (j & 1))) & 0xFFFF);
                const int scj = (int)(int8_t)(scw[(8 * H + j) >> 2] >> (8 * ((8 * H + j) & 3)));
                Ct[t] += scj * (dot[j] - 32 * bs);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; t++) acc[t] = fmaf(A.d[t * A.nbx + B] * D, (float)Ct[t], acc[t]);
}

// ---- one whole block per lane: Q8_0 (34 bytes, 2-byte aligned) ----
template <int NT>
__device__ __forceinline__ void blk_q8_0(const uint8_t* blk, int B, const ActView& A, float acc[NT]) {
    const float Dw = h2f_bits(*reinterpret_cast<const uint16_t*>(blk));
    uint32_t w[8];
    lds_words_any<8>(blk + 2, w);
#pragma unroll
    for (int t = 0; t < NT; t++) {
        const int8_t* xq = A.q + t * A.n_in;
        const uint4 x0 = *reinterpret_cast<const uint4*>(xq + q8_chunk(B, 0));
        const uint4 x1 = *reinterpret_cast<const uint4*>(xq + q8_chunk(B, 1));
        int I = dp4a(w[0], x0.x, 0);
        I = dp4a(w[1], x0.y, I);
        I = dp4a(w[2], x0.z, I);
        I = dp4a(w[3], x0.w, I);
        I = dp4a(w[4], x1.x, I);
        I = dp4a(w[5], x1.y, I);
        I = dp4a(w[6], x1.z, I);
        I = dp4a(w[7], x1.w, I);
        acc[t] = fmaf(Dw * A.d[t * A.nbx + B], (float)I, acc[t]);
    }
}

template <int NT>
__device__ __forceinline__ void block_dot(int type, const uint8_t* blk, int B, const ActView& A, float acc[NT]) {
    if (type == SYN_Q4_K) blk_q4_k<NT>(blk, B, A, acc);
    else if (type == SYN_Q6_K) blk_q6_k<NT>(blk, B, A, acc);
    else blk_q8_0<NT>(blk, B, A, acc);
}

// Position in a warp's range: matrix j, row, block column.  A stage is either whole rows
// or (rows wider than a stage) a run of blocks of one row.
struct Cursor {
    int j;
    int64_t row, rows_end;
    int bcol;
};

template <int NT>
__global__ void __launch_bounds__(GV_WARPS * 32, 1) k_gemv(const __grid_constant__ GemvBatch b) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * GV_WARPS + warp;
    const int GW = gridDim.x * GV_WARPS;
    uint8_t* ring = smem + b.off_stage + (size_t)warp * GV_NS * GV_SLOT;
    const uint32_t ring_addr = smem_u32(ring);
    const uint32_t bar0 = smem_u32(smem + b.off_bar) + warp * GV_NS * 8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + b.off_flag);

    if (threadIdx.x == 0) *abort_flag = 0;
    if (lane == 0)
        for (int s = 0; s < GV_NS; s++) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();

    // this warp's rows: from (j0, r0) up to (j1, r1), cut at row boundaries
    int j0, j1, ja, jb;
    int64_t r0, r1, ra, rb;
    row_at(b, b.total_bytes * gw / GW, j0, r0);
    row_at(b, b.total_bytes * (gw + 1) / GW, j1, r1);
    // the matrices any warp of this CTA touches (their activations are converted below)
    row_at(b, b.total_bytes * (blockIdx.x * GV_WARPS) / GW, ja, ra);
    row_at(b, b.total_bytes * ((blockIdx.x + 1) * GV_WARPS) / GW, jb, rb);
    if (rb == 0 && jb > ja) jb--;

    __syncthreads();

    // start of the range; skips matrices with no rows in it; false when empty
    auto begin = [&](Cursor& c) -> bool {
        c.j = j0;
        c.row = r0;
        c.bcol = 0;
        while (true) {
            c.rows_end = c.j == j1 ? r1 : b.job[c.j].n_out;
            if (c.row < c.rows_end) return true;
            if (c.j >= j1) return false;
            c.j++;
            c.row = 0;
        }
    };
    // blocks (and whole rows, or 0 for a run inside one row) of the stage at c
    auto extent = [&](const Cursor& c, int& nblk, int& nrows) {
        const GemvJob& J = b.job[c.j];
        if (J.stage_blocks >= J.nb) {
            nrows = (int)min((int64_t)(J.stage_blocks / J.nb), c.rows_end - c.row);
            nblk = nrows * J.nb;
        } else {
            nrows = 0;
            nblk = min(J.stage_blocks, J.nb - c.bcol);
        }
    };
    auto advance = [&](Cursor& c, int nblk, int nrows) -> bool {
        if (nrows > 0) {
            c.row += nrows;
        } else {
            c.bcol += nblk;
            if (c.bcol == b.job[c.j].nb) {
                c.bcol = 0;
                c.row++;
            }
        }
        while (c.row >= c.rows_end) {
            if (c.j >= j1) return false;
            c.j++;
            c.row = 0;
            c.bcol = 0;
            c.rows_end = c.j == j1 ? r1 : b.job[c.j].n_out;
        }
        return true;
    };

    // bulk copy of the stage at cursor c into ring slot s
    auto issue = [&](const Cursor& c, int nblk, uint32_t s) {
        const GemvJob& J = b.job[c.j];
        const int64_t src = (c.row * J.nb + c.bcol) * (int64_t)J.bb;
        const int64_t len = (int64_t)nblk * J.bb;
        const int64_t a0 = src & ~int64_t(15);
        if (lane == 0) {
            fence_proxy_async_smem();
            int64_t a1 = (src + len + 15) & ~int64_t(15);
            if (a1 > J.total_floor16) a1 = J.total_floor16;
            const uint32_t bytes = a1 > a0 ? (uint32_t)(a1 - a0) : 0u;
            const uint32_t bar = bar0 + 8 * s;
            mbar_arrive_expect_tx(bar, bytes);
            if (bytes) bulk_g2s(ring_addr + s * GV_SLOT, J.W + a0, bytes, bar);
        }
        if (src + len > J.total_floor16) {  // bytes past the last 16-byte boundary of W
            const int64_t from = J.total_floor16 > a0 ? J.total_floor16 : a0;
            for (int64_t k = from + lane; k < src + len; k += 32) ring[s * GV_SLOT + (k - a0)] = J.W[k];
            __syncwarp();
        }
    };

    uint32_t seq = 0;  // stage uses of this warp so far
    bool failed = false;
    for (int64_t t0 = 0; t0 < b.n_tok && !failed; t0 += NT) {
        // weights first: the copies are in flight while the activations are converted
        Cursor ic;
        bool more_i = begin(ic);
        uint32_t qi = seq;
        for (int k = 0; k < GV_NS - 1 && more_i; k++) {
            int nblk, nrows;
            extent(ic, nblk, nrows);
            issue(ic, nblk, (qi++) % GV_NS);
            more_i = advance(ic, nblk, nrows);
        }
        __syncthreads();  // every warp is done with the previous token group's activations
        act_to_smem<NT>(b, ja, jb, t0, smem);
        __syncthreads();
        if (*abort_flag) break;

        Cursor cc;
        bool more_c = begin(cc);
        float acc[NT];
#pragma unroll
        for (int t = 0; t < NT; t++) acc[t] = 0.f;
        uint32_t qc = seq;
        while (more_c) {
            if (more_i) {
                int nblk, nrows;
                extent(ic, nblk, nrows);
                __syncwarp();
                issue(ic, nblk, (qi++) % GV_NS);
                more_i = advance(ic, nblk, nrows);
            }
            const uint32_t s = qc % GV_NS;
            if (!mbar_wait(bar0 + 8 * s, (qc / GV_NS) & 1, b.err, abort_flag)) {
                // drain this warp's copies still in flight (bounded), so that no bulk copy
                // targets the shared memory of a finished CTA
                for (uint32_t k = qc; k < qi; k++) {
                    const long long w0 = clock64();
                    while (!mbar_try_wait(bar0 + 8 * (k % GV_NS), (k / GV_NS) & 1) &&
                           clock64() - w0 < SYN_WAIT_CYCLES / 8) {
                    }
                }
                failed = true;
                break;
            }
            qc++;
            const GemvJob& J = b.job[cc.j];
            const int type = J.type, nb = J.nb, bb = J.bb, lg = J.lg_nb;
            const ActView A{reinterpret_cast<const int8_t*>(smem + J.act_q),
                            reinterpret_cast<const float*>(smem + J.act_d),
                            reinterpret_cast<const int16_t*>(smem + J.act_s), J.n_in, J.nbx};
            float* Y = J.Y;
            const int64_t n_out = J.n_out;
            int nblk, nrows;
            extent(cc, nblk, nrows);
            if (nblk <= 0) {  // cannot happen with a valid geometry; never spin without progress
                failed = true;
                break;
            }
            const uint8_t* sbase = ring + s * GV_SLOT + (int)(((cc.row * nb + cc.bcol) * (int64_t)bb) & 15);
            if (lg >= 0) {
                // rows of 2^lg <= 32 blocks: 32 >> lg rows per warp step, lane = (row, block)
                for (int s0 = 0; s0 < nblk; s0 += 32) {
                    const int sidx = s0 + lane;
                    if (sidx < nblk) block_dot<NT>(type, sbase + sidx * bb, sidx & (nb - 1), A, acc);
#pragma unroll
                    for (int t = 0; t < NT; t++) {
                        const float v = group_sum(acc[t], lg);
                        if ((lane & (nb - 1)) == 0 && sidx < nblk && t0 + t < b.n_tok)
                            Y[(t0 + t) * n_out + cc.row + (sidx >> lg)] = v;
                        acc[t] = 0.f;
                    }
                }
            } else {
                // wider rows: each row (or run of one row) takes ceil(blocks / 32) warp steps
                const int per_row = nrows > 0 ? nb : nblk;
                const int rows = nrows > 0 ? nrows : 1;
                const int bstart = nrows > 0 ? 0 : cc.bcol;
                for (int r = 0; r < rows; r++) {
                    const uint8_t* rowp = sbase + (int64_t)r * nb * bb;
                    for (int s0 = 0; s0 < per_row; s0 += 32) {
                        const int kb = s0 + lane;
                        if (kb < per_row) block_dot<NT>(type, rowp + kb * bb, bstart + kb, A, acc);
                    }
                    if (nrows > 0 || cc.bcol + nblk == nb) {
#pragma unroll
                        for (int t = 0; t < NT; t++) {
                            const float v = warp_sum(acc[t]);
                            if (lane == 0 && t0 + t < b.n_tok) Y[(t0 + t) * n_out + cc.row + r] = v;
                            acc[t] = 0.f;
                        }
                    }
                }
            }
            __syncwarp();
            more_c = advance(cc, nblk, nrows);
        }
        seq = qi;
    }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------

static int64_t up16(int64_t v) { return (v + 15) & ~int64_t(15); }

// Shared memory left for the converted activations next to the weight rings.
static constexpr int64_t GEMV_ACT_BUDGET = (227 * 1024) - GV_WARPS * GV_NS * (GV_SLOT + 8) - 256;
static_assert(GEMV_ACT_BUDGET >= 8 * 1024, "decode ring leaves too little shared memory");
int64_t gemv_act_limit() { return GEMV_ACT_BUDGET; }

static int64_t act_bytes_per_token(int type, int64_t n_in) {
    if (type == SYN_Q8_0) return n_in + (n_in / 32) * 4;
    return n_in + (n_in / 256) * 4 + (n_in / 16) * 2;
}

template <int NT>
static cudaError_t run_gemv(GemvBatch& b, int sms, cudaStream_t s) {
    int64_t off = 0;
    for (int j = 0; j < b.n_jobs; j++) {
        GemvJob& J = b.job[j];
        J.act_q = (int)off;
        off = up16(off + (int64_t)NT * J.n_in);
        J.act_d = (int)off;
        off = up16(off + (int64_t)NT * J.nbx * 4);
        J.act_s = (int)off;
        off = up16(off + (J.type == SYN_Q8_0 ? 0 : (int64_t)NT * (J.n_in / 16) * 2));
    }
    off = (off + 127) & ~int64_t(127);
    b.off_stage = (int)off;
    off += (int64_t)GV_WARPS * GV_NS * GV_SLOT;
    b.off_bar = (int)off;
    off += GV_WARPS * GV_NS * 8;
    b.off_flag = (int)off;
    off += 16;
    const size_t smem = (size_t)off;
    if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
    auto kern = k_gemv<NT>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    kern<<<sms, GV_WARPS * 32, smem, s>>>(b);
    return cudaGetLastError();
}

// One matrix of a launch.  Rows of a power-of-two number of blocks up to 32 are packed
// several per warp step; the stage then holds a multiple of 32 blocks.  Wider rows: whole
// rows per stage when a row fits, else runs of a multiple of 32 blocks.
static void make_job(GemvJob& J, const GemvDesc& d, int64_t byte_begin) {
    J.W = static_cast<const uint8_t*>(d.W);
    J.X = d.X;
    J.Y = d.Y;
    J.type = d.type;
    J.n_out = d.n_out;
    J.n_in = (int)d.n_in;
    J.bb = block_bytes(d.type);
    J.nb = (int)(d.n_in / block_elems(d.type));
    J.row_bytes = (int64_t)J.nb * J.bb;
    J.total_floor16 = (d.n_out * J.row_bytes) & ~int64_t(15);
    J.byte_begin = byte_begin;
    J.nbx = (int)(d.n_in / (d.type == SYN_Q8_0 ? 32 : 256));
    const int fit = GV_STAGE / J.bb;  // >= 32 for every format
    J.lg_nb = -1;
    if (fit < 32) {  // excluded by the static_assert on GV_STAGE; kept as a guard
        J.stage_blocks = std::max(1, std::min(fit, J.nb));
    } else if (J.nb <= 32 && (J.nb & (J.nb - 1)) == 0) {
        int lg = 0;
        while ((1 << lg) < J.nb) lg++;
        J.lg_nb = lg;
        J.stage_blocks = (fit / 32) * 32;  // whole rows, whole warp steps
    } else if (J.nb <= fit) {
        J.stage_blocks = (fit / J.nb) * J.nb;  // whole rows
    } else {
        J.stage_blocks = (fit / 32) * 32;  // runs of one row
    }
}

int64_t gemv_act_bytes(int type, int64_t n_in) { return act_bytes_per_token(type, n_in) + 64; }

cudaError_t launch_gemv_batch(int n, const GemvDesc* d, int64_t n_tok, int* err, int sms, cudaStream_t s) {
    if (n < 1 || n > GEMV_MAX_JOBS) return cudaErrorInvalidValue;
    GemvBatch b{};
    b.n_jobs = n;
    b.n_tok = n_tok;
    b.err = err;
    int64_t bytes = 0, act = 0;
    for (int j = 0; j < n; j++) {
        make_job(b.job[j], d[j], bytes);
        bytes += d[j].n_out * b.job[j].row_bytes;
        act += gemv_act_bytes(d[j].type, d[j].n_in);
    }
    b.total_bytes = bytes;
    if (act > GEMV_ACT_BUDGET) return cudaErrorInvalidConfiguration;
    int nt = 1;
    while (nt < 8 && nt < n_tok && 2 * nt * act <= GEMV_ACT_BUDGET) nt *= 2;
    switch (nt) {
    case 1: return run_gemv<1>(b, sms, s);
    case 2: return run_gemv<2>(b, sms, s);
    case 4: return run_gemv<4>(b, sms, s);
    default: return run_gemv<8>(b, sms, s);
    }
}

cudaError_t launch_gemv(int type, const void* W, int64_t n_out, int64_t n_in, const float* X, int64_t n_tok,
                        float* Y, int* err, int sms, cudaStream_t s) {
    const GemvDesc d{type, W, n_out, n_in, X, Y};
    return launch_gemv_batch(1, &d, n_tok, err, sms, s);
}

}  // namespace syn

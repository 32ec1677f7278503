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
// Two launches per product group, chained by programmatic dependent launch:
//   0. k_act_decode converts the activation rows of every matrix of the launch (the encoder
//      of syn_quantize_activations) into a global workspace, in a swizzled layout: the
//      16-byte chunks of consecutive blocks land in different bank groups.
// k_gemv: one CTA per SM.  The warps of the grid are dealt to the matrices of the launch in
// proportion to their bytes; each warp streams a contiguous range of rows of one matrix.
//   1. Each warp starts its 1-D bulk copies (cp.async.bulk, completion on an mbarrier)
//      into its own 2-deep ring of shared-memory stages: a stage is a run of whole blocks,
//      copied through a window widened to 16-byte boundaries (so 34- and 210-byte blocks
//      need no alignment); bytes past the last 16-byte boundary of W come by plain loads.
//      It does so before waiting for the conversion launch, then releases the next launch
//      on the stream (whose own weight copies then overlap this launch's tail).
//   2. One thread bulk-copies the converted activations of the CTA's matrices into shared
//      memory.  When every CTA needs at most one conversion unit per warp (narrow inputs,
//      few tokens), there is no conversion launch: the CTA bulk-copies its fp32 activation
//      rows into shared memory and its warps run the encoder there (k_gemv<NT, true, FAM>).
//   3. Each lane decodes half a K-quant block or two 32-weight blocks per warp step: unpacks
//      4/5/6/8-bit codes in registers, forms the integer sub-block dots with dp4a, applies
//      the integer sub-block scales and then the fp32 block scales.  Rows of at most 32
//      blocks are spread over aligned groups of lanes, several rows per step; the partial
//      sums of a window of steps are reduced together (a transposed butterfly) and stored by
//      one coalesced store.  Wider rows take several steps and a whole-warp reduction.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "quant_dev.cuh"

namespace syn {

// Launch geometry (compile-time; the defaults are the measured best on GB300).
#ifndef SYN_GV_WARPS
#define SYN_GV_WARPS 16
#endif
#ifndef SYN_GV_NS
#define SYN_GV_NS 2
#endif
#ifndef SYN_GV_STAGE
#define SYN_GV_STAGE 4608
#endif
#ifndef SYN_GV_FAMILIES
#define SYN_GV_FAMILIES 1
#endif
#ifndef SYN_GV_LATE_UNITS
#define SYN_GV_LATE_UNITS 96
#endif
#ifndef SYN_GV_COST_Q6_K
#define SYN_GV_COST_Q6_K 130
#endif
#ifndef SYN_GV_COST_Q8_0
#define SYN_GV_COST_Q8_0 100
#endif
constexpr int GV_WARPS = SYN_GV_WARPS;
constexpr int GV_NS = SYN_GV_NS;            // stages per warp ring
// Launches whose conversion has at least this many units let the next launch on the stream
// start only when they end (see late_trigger).
constexpr int GV_LATE_UNITS = SYN_GV_LATE_UNITS;
constexpr int GV_STAGE = SYN_GV_STAGE;      // bytes of whole blocks per stage (at most)
constexpr int GV_SLOT = GV_STAGE + 32;      // stage slot: data plus the alignment window
constexpr int GV_MAX_SMS = 160;             // grid bound of the per-warp matrix table
// A stage must hold one warp step of every format: 16 blocks of Q4_K (144 bytes) or Q6_K
// (210 bytes, two lanes per block), 64 blocks of Q8_0 (34 bytes, two blocks per lane).
static_assert(GV_STAGE >= 16 * 210 && GV_STAGE >= 64 * 34, "decode stage smaller than one warp step");

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
    int bps;                // blocks per warp step: 16 (Q4_K, Q6_K: two lanes per block), 64 (Q8_0)
    int lg_nb;              // log2(nb) when rows are packed several per warp step, else -1
    int nbx;                // activation blocks per row
    int units;              // conversion-kernel units (warp steps) per token
    int act_src;            // the job whose converted activations this one reads: itself, or
                            // the first job of the launch with the same input (X, n_in and
                            // activation layout), which converts it once for both
    int warp_begin, warp_end;  // the decode warps of this matrix
    int upr;                // work units per row: 1 (whole rows), or 2 for rows of two stages
                            // runs: the two runs may go to different warps and are then added
                            // into Y (zeroed by the conversion kernel; a sum of two partials
                            // onto zero does not depend on their order)
    int n_units;            // n_out * upr
    int ds;                 // per-token stride of the activation scales (floats, multiple of 4)
    int act_q, act_d, act_s;  // shared-memory offsets of the converted activations (NT tokens)
    uint8_t* actg;          // the same, for all n_tok tokens, in the global workspace:
    int64_t g_d, g_s;       //   codes at actg, scales at actg + g_d, 16-sums at actg + g_s
};

struct GemvBatch {
    GemvJob job[GEMV_MAX_JOBS];
    int n_jobs;
    int64_t total_bytes;
    int64_t n_tok;
    int* err;
    int fused;              // 1: each CTA converts its own activations (no conversion launch)
    int off_x;              // fused: shared-memory staging of the CTA's fp32 activation rows
    int off_stage, off_bar, off_flag;
    int late_trigger;       // 1: the next launch starts only when this one has ended.  A large
                            // conversion of the next step (a layer like this one) would
                            // otherwise crowd its CTAs onto the first SMs this launch frees
                            // and run there compute-bound; started after the end, they spread
    int n_conv;             // conversion launch: one row of CTAs per listed job (the jobs that
    uint8_t conv_job[GEMV_MAX_JOBS];  // convert their input, or whose Y must be zeroed)
    // matrix of each decode warp of the grid: one parameter-space load instead of a
    // dependent walk over the job table
    uint8_t warp_job[GV_MAX_SMS * GV_WARPS];
    // per CTA, bit j: the CTA copies (or converts) job j's activations, i.e. j is the first
    // of the CTA's jobs to read them
    uint16_t act_mask[GV_MAX_SMS];
};

// Bytes of dynamic shared memory this launch was given.
__device__ __forceinline__ uint32_t dyn_smem_bytes() {
    uint32_t v;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Whether job j is the first of jobs ja..j to read its converted activations (the one that
// copies or converts them for the CTA); host side, for the per-CTA masks.
static bool first_reader(const GemvBatch& b, int ja, int j) {
    for (int i = ja; i < j; i++)
        if (b.job[i].act_src == b.job[j].act_src) return false;
    return true;
}

// Sum over aligned groups of 2^lg lanes (lg <= 5).
// Window of packed warp steps whose row sums are reduced together: 8 / NT steps.
template <int NT>
struct Win {
    static constexpr int N = NT >= 8 ? 1 : 8 / NT;
};

// Rows of at most 32 blocks: every warp step leaves, in each aligned group of 2^lgl lanes,
// the partial sums of one row.  The partials of the last Win steps are kept (part[i] is step
// i of the window; a window of n < N steps sits in part[N - n ..]) and reduced at once: a
// transposed butterfly over the group (offsets 2^(lgl-1) .. 1) that, while a lane holds more
// than one value, sends half of them to its partner and keeps the other half; then plain
// butterfly steps.  Each row's partials are added in the same tree whatever the window, so
// the result does not depend on where a row falls.  The one lane per group and value that
// holds a total writes it: rows row0 + step * rstep + (lane >> lgl), rows below row_end.
template <int NT>
__device__ __forceinline__ void win_flush(float (&part)[Win<NT>::N][NT], int n, int lgl, int lane, int64_t row0,
                                          int rstep, int64_t row_end, float* Y, int64_t n_out, int64_t t0,
                                          int64_t n_tok) {
    constexpr int N = Win<NT>::N;
    if (N > 1 && n == 1) {  // one step: the plain butterfly on it alone (same tree per row)
        const int64_t row = row0 + (lane >> lgl);
#pragma unroll
        for (int t = 0; t < NT; t++) {
            float v = part[N - 1][t];
            for (int k = 0; k < lgl; k++) v += __shfl_xor_sync(0xffffffffu, v, 1 << (lgl - 1 - k));
            if ((lane & ((1 << lgl) - 1)) == 0 && row < row_end && t0 + t < n_tok && SYN_IN_BOUNDS(row < n_out))
                Y[(t0 + t) * n_out + row] = v;
            part[N - 1][t] = 0.f;
        }
        return;
    }
    int vbase = 0, k_done = 0;
#pragma unroll
    for (int k = 0; (N >> k) > 1; k++) {
        if (k < lgl) {
            const int o = 1 << (lgl - 1 - k);
            const bool up = (lane & o) != 0;
            const int half = N >> (k + 1);
#pragma unroll
            for (int i = 0; i < (N >> (k + 1)); i++) {
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    const float send = up ? part[i][t] : part[i + half][t];
                    const float keep = up ? part[i + half][t] : part[i][t];
                    part[i][t] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            if (up) vbase += half;
            k_done = k + 1;
        }
    }
    for (int k = k_done; k < lgl; k++) {
        const int o = 1 << (lgl - 1 - k);
#pragma unroll
        for (int t = 0; t < NT; t++) part[0][t] += __shfl_xor_sync(0xffffffffu, part[0][t], o);
    }
    const int left = N >> k_done;  // values this lane holds
    const bool writer = (lane & ((1 << (lgl - k_done)) - 1)) == 0;
#pragma unroll
    for (int i = 0; i < N; i++) {
        if (i < left && writer) {
            const int step = vbase + i - (N - n);
            const int64_t row = row0 + (int64_t)step * rstep + (lane >> lgl);
            if (step >= 0 && row < row_end && SYN_IN_BOUNDS(row < n_out)) {
#pragma unroll
                for (int t = 0; t < NT; t++)
                    if (t0 + t < n_tok) Y[(t0 + t) * n_out + row] = part[i][t];
            }
        }
    }
#pragma unroll
    for (int i = 0; i < N; i++)
#pragma unroll
        for (int t = 0; t < NT; t++) part[i][t] = 0.f;
}

// Swizzled activation chunks: byte offset of chunk c (16 bytes) of block B.  The two lanes
// of a K-quant block read chunks c and c + 8 of it, and the four blocks of a quarter-warp
// are consecutive: chunk c of block B goes to 16-byte bank group (c ^ B ^ 4*(c >= 8)) % 8,
// so the eight 16-byte reads of a quarter-warp fall in eight different bank groups.
__device__ __forceinline__ int k_chunk(int B, int c) { return 256 * B + 16 * (c ^ (B & 7) ^ ((c >> 3) << 2)); }
__device__ __forceinline__ int q8_chunk(int B, int c) { return 32 * B + 16 * (c ^ ((B >> 2) & 1)); }

// Activation sums per token, in int16 elements (the per-token stride): the 16-sums for the
// K-quants (n_in/16 of them), one code sum per 32-block for Q4_0 / Q5_0 (their codes carry
// an offset), padded to 8 so that every token's sums start on 16 bytes; none for Q8_0.
__host__ __device__ __forceinline__ int64_t sum_stride(int type, int64_t n_in) {
    return type == SYN_Q8_0 ? 0 : small_block(type) ? ((n_in / 32 + 7) & ~int64_t(7)) : n_in / 16;
}
__host__ __device__ __forceinline__ int64_t sum_bytes(int type, int64_t n_in) { return 2 * sum_stride(type, n_in); }

// Conversion unit r of matrix J: token r / units, then a 256-block (K-quants, 8 values per
// lane) or four 32-blocks (the Q8_0 family, 4 values per lane; blocks past the row are 0).
// Token r / units is row r / units of X (n_in floats each).  unit_load reads the lane's
// values, unit_store encodes them into the decode layout (codes with swizzled 16-byte chunks,
// block scales, 16-sums (K-quants) or block code sums (Q4_0 / Q5_0)) at slot r / units.
// One warp.
__device__ __forceinline__ void unit_load(const GemvJob& J, const float* X, int r, int lane, float v[8]) {
    if (small_block(J.type)) {
        const int t = r / J.units;
        const int blk = (r - t * J.units) * 4 + (lane >> 3), e = lane & 7;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (blk < J.nbx) x = *reinterpret_cast<const float4*>(X + (int64_t)t * J.n_in + blk * 32 + 4 * e);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        v[4] = v[5] = v[6] = v[7] = 0.f;
    } else {
        const int t = r / J.nbx;
        const int blk = r - t * J.nbx;
        const float* x = X + (int64_t)t * J.n_in + blk * 256 + lane * 8;
        const float4 x0 = *reinterpret_cast<const float4*>(x);
        const float4 x1 = *reinterpret_cast<const float4*>(x + 4);
        v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
        v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
    }
}

__device__ __forceinline__ void unit_store(const GemvJob& J, int r, const float v[8], int8_t* aq, float* ad, int16_t* as,
                                           int lane) {
    bool fin;
    if (small_block(J.type)) {
        const int t = r / J.units;
        const int blk = (r - t * J.units) * 4 + (lane >> 3), e = lane & 7;
        uint16_t db;
        const uint32_t q = q8_0_group(v, &db, &fin);
        // Q4_0 / Q5_0 weights: the block's code sum, for the -8 / -16 offset of their codes
        int qs = 0;
        if (J.type != SYN_Q8_0) {
            qs = __dp4a((int)q, 0x01010101, 0);
            qs += __shfl_xor_sync(0xffffffffu, qs, 1);
            qs += __shfl_xor_sync(0xffffffffu, qs, 2);
            qs += __shfl_xor_sync(0xffffffffu, qs, 4);
        }
        if (blk < J.nbx) {
            *reinterpret_cast<uint32_t*>(aq + (int64_t)t * J.n_in + q8_chunk(blk, e >> 2) + 4 * (e & 3)) = q;
            if (e == 0) ad[(int64_t)t * J.ds + blk] = h2f_bits(db);
            if (e == 0 && J.type != SYN_Q8_0) as[(int64_t)t * sum_stride(J.type, J.n_in) + blk] = (int16_t)qs;
        }
    } else {
        const int t = r / J.nbx;
        const int blk = r - t * J.nbx;
        uint32_t w0, w1;
        float dd;
        int bs;
        q8_k_warp(v, &w0, &w1, &dd, &bs, &fin);
        *reinterpret_cast<uint2*>(aq + (int64_t)t * J.n_in + k_chunk(blk, lane >> 1) + 8 * (lane & 1)) =
            make_uint2(w0, w1);
        if (lane == 0) ad[(int64_t)t * J.ds + blk] = dd;
        if ((lane & 1) == 0) as[((int64_t)t * J.nbx + blk) * 16 + (lane >> 1)] = (int16_t)bs;
    }
}

// Convert every activation row of every matrix of the launch into the global workspace,
// in the layout the decode kernel copies to shared memory.  One row of CTAs per matrix.
// Lets the dependent decode launch start (programmatic dependent launch) at once.  It is
// itself launched as a programmatic dependent of whatever precedes it on the stream, so it
// waits for that work (which may produce X, or still read the workspace and Y this kernel
// writes) before touching memory.
__global__ void __launch_bounds__(128) k_act_decode(const __grid_constant__ GemvBatch b) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int GW = (int)((gridDim.x * blockDim.x) >> 5);
    // 32-bit index arithmetic only (64-bit division runs on the slow fp64 pipe)
    const int j = b.conv_job[blockIdx.y];
    const GemvJob& J = b.job[j];
    if (J.upr > 1) {  // runs of this matrix's rows are added into Y by different warps
        const int ny = (int)b.n_tok * (int)J.n_out;
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < ny; i += gridDim.x * blockDim.x) J.Y[i] = 0.f;
    }
    if (J.act_src != j) return;  // its input is converted by the job it shares it with
    const int n_units = (int)b.n_tok * J.units;
    for (int r = gw; r < n_units; r += GW)
    {
        float v[8];
        unit_load(J, J.X, r, lane, v);
        unit_store(J, r, v, reinterpret_cast<int8_t*>(J.actg), reinterpret_cast<float*>(J.actg + J.g_d),
                   reinterpret_cast<int16_t*>(J.actg + J.g_s), lane);
    }
}

struct ActView {
    const int8_t* q;    // token 0 codes (swizzled chunks); token t at + t * n_in
    const float* d;     // token 0 scales; token t at + t * ds
    const int16_t* s;   // token 0 sums (K-quants: 16-sums, Q4_0/Q5_0: block code sums);
                        // token t at + t * sst
    int n_in, nbx, ds, sst;
};

// ---- Q4_K: half a block per lane (h = 0: sub-blocks 0..3, h = 1: sub-blocks 4..7) ----
// blk is 16-byte aligned in shared memory (144-byte blocks, 16-byte aligned rows).
template <int NT>
__device__ __forceinline__ void lane_q4_k(const uint8_t* blk, int h, int B, const ActView& A, float acc[NT]) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const float D = h2f_bits(hdr.x & 0xFFFF), Dm = h2f_bits(hdr.x >> 16);
    // the 6-bit scales and mins of sub-blocks 4h .. 4h+3, one per byte (all four at once)
    const uint32_t scw = h ? ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u)) : (hdr.y & 0x3F3F3F3Fu);
    const uint32_t mnw = h ? (((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u)) : (hdr.z & 0x3F3F3F3Fu);
    int At[NT];
#pragma unroll
    for (int t = 0; t < NT; t++) At[t] = 0;
#pragma unroll
    for (int cc = 0; cc < 2; cc++) {  // code chunk c = 2h + cc: sub-blocks 2c (low), 2c+1 (high)
        const int c = 2 * h + cc;
        const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
        const uint32_t q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const int sl = (int)__byte_perm(scw, 0, 0x4440 | (2 * cc)), sh = (int)__byte_perm(scw, 0, 0x4441 | (2 * cc));
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const int8_t* xq = A.q + t * A.n_in;
            const uint4 x0 = *reinterpret_cast<const uint4*>(xq + k_chunk(B, 4 * c));
            const uint4 x1 = *reinterpret_cast<const uint4*>(xq + k_chunk(B, 4 * c + 1));
            const uint4 x2 = *reinterpret_cast<const uint4*>(xq + k_chunk(B, 4 * c + 2));
            const uint4 x3 = *reinterpret_cast<const uint4*>(xq + k_chunk(B, 4 * c + 3));
            const uint32_t xl[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const uint32_t xh[8] = {x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
            int dl = 0, dh16 = 0;  // dh16: 16 x the high-nibble dot (nibbles masked in place)
#pragma unroll
            for (int i = 0; i < 8; i++) {
                dl = dp4a(q[i] & 0x0F0F0F0Fu, xl[i], dl);
                dh16 = dp4a_us(q[i] & 0xF0F0F0F0u, xh[i], dh16);
            }
            At[t] += sl * dl + sh * (dh16 >> 4);
        }
    }
    // min term: sum_j m_j * (16-sum 2j + 16-sum 2j+1) of sub-blocks 4h+j, as four 16x8-bit
    // dot products (dp2a) against the mins duplicated per byte pair
    const int m01 = (int)__byte_perm(mnw, 0, 0x1100), m23 = (int)__byte_perm(mnw, 0, 0x3322);
#pragma unroll
    for (int t = 0; t < NT; t++) {
        const uint4 sv = *reinterpret_cast<const uint4*>(A.s + (t * A.nbx + B) * 16 + 8 * h);
        int Bm = __dp2a_lo((int)sv.x, m01, 0);
        Bm = __dp2a_hi((int)sv.y, m01, Bm);
        Bm = __dp2a_lo((int)sv.z, m23, Bm);
        Bm = __dp2a_hi((int)sv.w, m23, Bm);
        acc[t] = fmaf(A.d[t * A.ds + B], D * (float)At[t] - Dm * (float)Bm, acc[t]);
    }
}

// ---- Q6_K: half a block per lane (weights 128H .. 128H+127); blk 2-byte aligned ----
// TOK_INNER: each sub-block's codes merged once and dotted with every token in turn (the
// Q6_K-only instantiation: lm_head 1-2 % faster); else token by token over the whole half
// (the mixed instantiation, where that order measured ~1 % faster).  The integer sums are the
// same either way, so are the results.
template <int NT, bool TOK_INNER>
__device__ __forceinline__ void lane_q6_k(const uint8_t* blk, int H, int B, const ActView& A, float acc[NT]) {
    const float D = h2f_bits(*reinterpret_cast<const uint16_t*>(blk + 208));
    uint32_t scw[2], ql[16], qh[8];
    lds_words_any<2>(blk + 192 + 8 * H, scw);  // int8 scales of sub-blocks 8H .. 8H+7
    lds_words_any<16>(blk + 64 * H, ql);
    lds_words_any<8>(blk + 128 + 32 * H, qh);
    // sub-block j's scale, sign-extended
    int scj[8];
#pragma unroll
    for (int j = 0; j < 8; j++) scj[j] = (int)(int8_t)(scw[j >> 2] >> (8 * (j & 3)));
    // codes (q + 32) of words w = 4*half + i of quarter k of the half: sub-block 8H + 2k + half
    auto codes = [&](int k, int w) {
        const uint32_t a = (k & 1) ? ql[8 + w] : ql[w];
        const uint32_t lo = (k >= 2) ? ((a >> 4) & 0x0F0F0F0Fu) : (a & 0x0F0F0F0Fu);
        const uint32_t hi = (k >= 2 ? (qh[w] >> (2 * k - 4)) : (qh[w] << (4 - 2 * k))) & 0x30303030u;
        return lo | hi;
    };
    int C[NT];
#pragma unroll
    for (int t = 0; t < NT; t++) C[t] = 0;
    if constexpr (TOK_INNER) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
#pragma unroll
            for (int half = 0; half < 2; half++) {
                const int j = 2 * k + half;
                uint32_t q[4];
#pragma unroll
                for (int i = 0; i < 4; i++) q[i] = codes(k, 4 * half + i);
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    const uint4 x = *reinterpret_cast<const uint4*>(A.q + t * A.n_in + k_chunk(B, 8 * H + j));
                    int dsum = dp4a(q[0], x.x, 0);
                    dsum = dp4a(q[1], x.y, dsum);
                    dsum = dp4a(q[2], x.z, dsum);
                    dsum = dp4a(q[3], x.w, dsum);
                    C[t] += scj[j] * dsum;
                }
            }
        }
    } else {
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const int8_t* xq = A.q + t * A.n_in;
#pragma unroll
            for (int k = 0; k < 4; k++) {
#pragma unroll
                for (int half = 0; half < 2; half++) {
                    const int j = 2 * k + half;
                    const uint4 x = *reinterpret_cast<const uint4*>(xq + k_chunk(B, 8 * H + j));
                    const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
                    int dsum = 0;
#pragma unroll
                    for (int i = 0; i < 4; i++) dsum = dp4a(codes(k, 4 * half + i), xw[i], dsum);
                    C[t] += scj[j] * dsum;
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; t++) {
        // the stored codes are q + 32: subtract 32 * sum_j sc_j * (16-sum j), by dp2a
        const uint4 sv = *reinterpret_cast<const uint4*>(A.s + (t * A.nbx + B) * 16 + 8 * H);
        int SB = __dp2a_lo((int)sv.x, (int)scw[0], 0);
        SB = __dp2a_hi((int)sv.y, (int)scw[0], SB);
        SB = __dp2a_lo((int)sv.z, (int)scw[1], SB);
        SB = __dp2a_hi((int)sv.w, (int)scw[1], SB);
        acc[t] = fmaf(A.d[t * A.ds + B] * D, (float)(C[t] - 32 * SB), acc[t]);
    }
}

// ---- Q8_0: n (1 or 2) consecutive 34-byte blocks per lane; blk 2-byte aligned ----
template <int NT>
__device__ __forceinline__ void lane_q8_0(const uint8_t* blk, int n, int B, const ActView& A, float acc[NT]) {
#pragma unroll
    for (int e = 0; e < 2; e++) {
        if (e >= n) break;
        const uint8_t* p = blk + 34 * e;
        const float Dw = h2f_bits(*reinterpret_cast<const uint16_t*>(p));
        uint32_t w[8];
        lds_words_any<8>(p + 2, w);
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const int8_t* xq = A.q + t * A.n_in;
            const uint4 x0 = *reinterpret_cast<const uint4*>(xq + q8_chunk(B + e, 0));
            const uint4 x1 = *reinterpret_cast<const uint4*>(xq + q8_chunk(B + e, 1));
            int I = dp4a(w[0], x0.x, 0);
            I = dp4a(w[1], x0.y, I);
            I = dp4a(w[2], x0.z, I);
            I = dp4a(w[3], x0.w, I);
            I = dp4a(w[4], x1.x, I);
            I = dp4a(w[5], x1.y, I);
            I = dp4a(w[6], x1.z, I);
            I = dp4a(w[7], x1.w, I);
            acc[t] = fmaf(Dw * A.d[t * A.ds + B + e], (float)I, acc[t]);
        }
    }
}

// ---- Q4_0 / Q5_0 (OFF = 8 / 16): n (1 or 2) consecutive 18- / 22-byte blocks per lane;
// blk 2-byte aligned.  I = sum q*x - OFF * (sum of the activation codes of the block). ----
template <int NT, int OFF>
__device__ __forceinline__ void lane_qx_0(const uint8_t* blk, int n, int B, const ActView& A, float acc[NT]) {
    constexpr int BB = OFF == 8 ? 18 : 22;
#pragma unroll
    for (int e = 0; e < 2; e++) {
        if (e >= n) break;
        const uint8_t* p = blk + BB * e;
        const float Dw = h2f_bits(*reinterpret_cast<const uint16_t*>(p));
        uint32_t w[5];
        if (OFF == 8) lds_words_any<4>(p + 2, w + 1);
        else lds_words_any<5>(p + 2, w);  // w[0] = qh: bit k = fifth bit of code k
        // codes 4i..4i+3 and 16+4i..16+4i+3, one per byte (Q4_0: the high nibbles masked in
        // place, 16 x the code, their dot divided by 16 afterwards, exactly)
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            lo[i] = w[1 + i] & 0x0F0F0F0Fu;
            hi[i] = OFF == 8 ? (w[1 + i] & 0xF0F0F0F0u) : ((w[1 + i] >> 4) & 0x0F0F0F0Fu);
            if (OFF == 16) {  // spread 4 bits of qh into bit 4 of 4 bytes
                lo[i] |= ((((w[0] >> (4 * i)) & 15u) * 0x00204081u) & 0x01010101u) << 4;
                hi[i] |= ((((w[0] >> (16 + 4 * i)) & 15u) * 0x00204081u) & 0x01010101u) << 4;
            }
        }
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const int8_t* xq = A.q + t * A.n_in;
            const uint4 x0 = *reinterpret_cast<const uint4*>(xq + q8_chunk(B + e, 0));
            const uint4 x1 = *reinterpret_cast<const uint4*>(xq + q8_chunk(B + e, 1));
            int I = dp4a(lo[0], x0.x, 0);
            I = dp4a(lo[1], x0.y, I);
            I = dp4a(lo[2], x0.z, I);
            I = dp4a(lo[3], x0.w, I);
            if (OFF == 8) {
                int H = dp4a_us(hi[0], x1.x, 0);
                H = dp4a_us(hi[1], x1.y, H);
                H = dp4a_us(hi[2], x1.z, H);
                H = dp4a_us(hi[3], x1.w, H);
                I += H >> 4;
            } else {
                I = dp4a(hi[0], x1.x, I);
                I = dp4a(hi[1], x1.y, I);
                I = dp4a(hi[2], x1.z, I);
                I = dp4a(hi[3], x1.w, I);
            }
            I -= OFF * (int)A.s[t * A.sst + B + e];
            acc[t] = fmaf(Dw * A.d[t * A.ds + B + e], (float)I, acc[t]);
        }
    }
}

// This lane's share of warp step `first` .. of a run of blocks: K-quants take half a block
// per lane (block first + lane/2, part lane%2); the 32-weight formats take two blocks per lane.
// `avail` = blocks of the run from `first` on; the activation block of run block i is
// (B0 + i) & bmask (bmask = nb - 1 when the run holds several whole rows).
// FAM: the formats the kernel instantiation handles (0: all; 2: the 32-weight formats; 3: Q4_K;
// 4: Q6_K), so that a launch of one format runs code without the others' lanes (measured:
// Llama-8B Q4_K layer 23.6 -> 23.0 us, Q6_K lm_head 78.8 -> 77.2 us; launches mixing Q4_K and
// Q6_K ran slower on a K-quant-only instantiation than on the general one, and keep it).
template <int NT, int FAM>
__device__ __forceinline__ void lane_step(int type, const uint8_t* base, int bb, int first, int avail, int B0,
                                          int bmask, const ActView& A, float acc[NT]) {
    const int lane = threadIdx.x & 31;
    if (FAM == 2 || (FAM == 0 && small_block(type))) {
        const int k = 2 * lane;
        if (k < avail) {
            const uint8_t* p = base + (first + k) * bb;
            const int n = min(2, avail - k), B = (B0 + k) & bmask;
            if (type == SYN_Q8_0) lane_q8_0<NT>(p, n, B, A, acc);
            else if (type == SYN_Q4_0) lane_qx_0<NT, 8>(p, n, B, A, acc);
            else lane_qx_0<NT, 16>(p, n, B, A, acc);
        }
    } else {
        const int k = lane >> 1;
        if (k < avail) {
            const int B = (B0 + k) & bmask;
            if (FAM == 3 || (FAM != 4 && type == SYN_Q4_K)) lane_q4_k<NT>(base + (first + k) * bb, lane & 1, B, A, acc);
            else lane_q6_k<NT, FAM == 4>(base + (first + k) * bb, lane & 1, B, A, acc);
        }
    }
}

// The warps of the grid are dealt to the matrices so that the largest per-warp byte count is
// as small as it can be (computed on the host into warp_job); a matrix's work units (rows, or
// runs of rows wider than a stage) are split evenly among its warps.  Returns this warp's
// matrix and units [u0, u1) (empty when the matrix has fewer units than warps).  32-bit
// arithmetic only: 64-bit division runs on the (slow) fp64 pipe.
__device__ __forceinline__ void warp_share(const GemvBatch& b, int gw, int& j, int& u0, int& u1) {
    j = b.warp_job[gw];
    const int nw = b.job[j].warp_end - b.job[j].warp_begin, i = gw - b.job[j].warp_begin;
    const int n = b.job[j].n_units, q = n / nw, rem = n - q * nw;
    u0 = q * i + (rem * i) / nw;
    u1 = q * (i + 1) + (rem * (i + 1)) / nw;
}

// FUSED: the CTA converts its activations itself (b.fused); a separate instantiation, so that
// the other path compiles as if it did not exist.
template <int NT, bool FUSED, int FAM>
__global__ void __launch_bounds__(GV_WARPS * 32, 1) k_gemv(const __grid_constant__ GemvBatch b) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * GV_WARPS + warp;
    uint8_t* ring = smem + b.off_stage + (size_t)warp * GV_NS * GV_SLOT;
    const uint32_t ring_addr = smem_u32(ring);
    const uint32_t bar0 = smem_u32(smem + b.off_bar) + warp * GV_NS * 8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + b.off_flag);

    const uint32_t act_bar = smem_u32(smem + b.off_flag + 8);
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(act_bar, 1);
    }
    if (lane == 0)
        for (int s = 0; s < GV_NS; s++) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();

    // this warp's matrix and rows; the matrices of the CTA's first and last warps bound
    // the activations the CTA converts
    int jw, u0, u1;
    warp_share(b, gw, jw, u0, u1);
    // this warp's units are units of its matrix (a failed check leaves the warp without work)
    if (!SYN_IN_BOUNDS(jw >= 0 && jw < b.n_jobs && u0 >= 0 && u0 <= u1 && u1 <= b.job[jw].n_units)) {
        jw = 0;
        u1 = u0 = 0;
    }
    const int ja = b.warp_job[blockIdx.x * GV_WARPS], jb = b.warp_job[blockIdx.x * GV_WARPS + GV_WARPS - 1];
    const uint32_t act_mask = b.act_mask[blockIdx.x];
    __syncthreads();

    // the matrix, in registers for the whole launch
    const GemvJob& Jp = b.job[jw];
    const uint8_t* const W = Jp.W;
    float* const Y = Jp.Y;
    const int64_t n_out = Jp.n_out, total_floor16 = Jp.total_floor16;
    const int type = Jp.type, nb = Jp.nb, bb = Jp.bb, lg = Jp.lg_nb, bps = Jp.bps;
    const int sblk = Jp.stage_blocks;
    const int rps = sblk >= nb ? sblk / nb : 0;  // whole rows per stage (0: runs of one row)
    const int upr = Jp.upr;
    const bool split = upr > 1;                   // each run is a unit, added into Y
    // first row and block column of this warp's units; units end at u1
    const int64_t r0 = split ? u0 / upr : u0;
    const int b0 = split ? (u0 - (u0 / upr) * upr) * sblk : 0;
    const int64_t r1 = u1;  // unsplit matrices: units are rows
    const ActView A{reinterpret_cast<const int8_t*>(smem + Jp.act_q), reinterpret_cast<const float*>(smem + Jp.act_d),
                    reinterpret_cast<const int16_t*>(smem + Jp.act_s), Jp.n_in, Jp.nbx, Jp.ds,
                    (int)sum_stride(type, Jp.n_in)};

    // stage extent at (row, bcol): blocks and whole rows (0 for a run inside one row)
    auto extent = [&](int64_t row, int bcol, int& nblk, int& nrows) {
        if (rps > 0) {
            nrows = (int)min((int64_t)rps, r1 - row);  // whole-row matrices only
            nblk = nrows * nb;
        } else {
            nrows = 0;
            nblk = min(sblk, nb - bcol);
        }
    };
    auto advance = [&](int64_t& row, int& bcol, int nblk, int nrows) {
        if (nrows > 0) {
            row += nrows;
        } else {
            bcol += nblk;
            if (bcol == nb) {
                bcol = 0;
                row++;
            }
        }
    };
    // bulk copy of the stage at (row, bcol) into ring slot s
    auto issue = [&](int64_t row, int bcol, int nblk, uint32_t s) {
        const int64_t src = (row * nb + bcol) * (int64_t)bb;
        const int64_t len = (int64_t)nblk * bb;
        const int64_t a0 = src & ~int64_t(15);
        // the stage's blocks lie inside W, and with their 16-byte window inside the slot
        const bool in = SYN_IN_BOUNDS(row >= 0 && nblk > 0 && src + len <= n_out * (int64_t)nb * bb &&
                                      (int)(src & 15) + len <= GV_SLOT);
        if (lane == 0) {
            fence_proxy_async_smem();
            int64_t a1 = (src + len + 15) & ~int64_t(15);
            if (a1 > total_floor16) a1 = total_floor16;
            const uint32_t bytes = in && a1 > a0 ? (uint32_t)(a1 - a0) : 0u;
            const uint32_t bar = bar0 + 8 * s;
            mbar_arrive_expect_tx(bar, bytes);
            if (bytes) bulk_g2s(ring_addr + s * GV_SLOT, W + a0, bytes, bar);
        }
        if (in && src + len > total_floor16) {  // bytes past the last 16-byte boundary of W
            const int64_t from = total_floor16 > a0 ? total_floor16 : a0;
            for (int64_t k = from + lane; k < src + len; k += 32) ring[s * GV_SLOT + (k - a0)] = W[k];
            __syncwarp();
        }
    };

    // After a wait gave up: the weight stages this warp issued and has not consumed, and
    // (thread 0, which issued them) the activation copies of the current token group land
    // before the CTA can leave, so that no bulk copy writes into the next CTA's shared memory.
    auto drain = [&](uint32_t from, uint32_t to, bool act_pending, uint32_t act_parity) {
        for (uint32_t k = from; k < to; k++) mbar_drain(bar0 + 8 * (k % GV_NS), (k / GV_NS) & 1, b.err);
        if (act_pending && threadIdx.x == 0) mbar_drain(act_bar, act_parity, b.err);
    };
#ifdef SYN_TEST_STALL
    constexpr bool act_issued = false;  // timeout-test build: the activation copies never come
#else
    constexpr bool act_issued = true;
#endif

    uint32_t seq = 0;  // stage uses of this warp so far
    bool failed = false;
    for (int64_t t0 = 0; t0 < b.n_tok && !failed; t0 += NT) {
        // weights first: the copies are in flight while the activations are converted
        int64_t irow = r0;
        int ibcol = b0;
        int iu = u0;  // units issued so far (rows, or runs of split matrices)
        uint32_t qi = seq;
        auto more = [&](int64_t row, int u) { return split ? u < u1 : row < r1; };
        for (int k = 0; k < GV_NS - 1 && more(irow, iu); k++) {
            int nblk, nrows;
            extent(irow, ibcol, nblk, nrows);
            issue(irow, ibcol, nblk, (qi++) % GV_NS);
            advance(irow, ibcol, nblk, nrows);
            iu++;
        }
        // the next launch on the stream may start now (a following conversion kernel waits
        // for this launch to finish before it touches memory; its own decode launch then
        // streams weights while this one drains), unless this launch's conversion is large
        // (late_trigger: the next one then starts when this launch ends)
        if (!b.late_trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // the converted activations of tokens t0.. of the CTA's matrices: written by the
        // conversion kernel this launch depends on, so wait for it first
        asm volatile("griddepcontrol.wait;" ::: "memory");
        __syncthreads();  // every warp is done with the previous token group's activations
        const uint32_t act_parity = (uint32_t)((t0 / NT) & 1);
        if (FUSED) {
            // the fp32 rows of tokens t0.. of the CTA's matrices by bulk copy into the staging
            // area, then converted by the CTA's warps (units dealt round-robin over matrices
            // ja..jb) into the activation layout
            const int nt = (int)min((int64_t)NT, b.n_tok - t0);
            if (threadIdx.x == 0 && act_issued) {
                uint32_t tx = 0;
                for (int j = ja; j <= jb; j++)
                    if ((act_mask >> j) & 1) tx += (uint32_t)(nt * b.job[j].n_in * 4);
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(act_bar, tx);
                uint32_t xo = 0;
                for (int j = ja; j <= jb; j++) {
                    if (!((act_mask >> j) & 1)) continue;
                    const GemvJob& J = b.job[j];
                    const uint32_t by = (uint32_t)(nt * J.n_in * 4);
                    // the staging area holds the rows (a failed check leaves the phase short:
                    // the wait for it then runs out)
                    if (SYN_IN_BOUNDS((uint32_t)b.off_x + xo + by <= dyn_smem_bytes()))
                        bulk_g2s(smem_u32(smem + b.off_x + xo), J.X + t0 * J.n_in, by, act_bar);
                    xo += by;
                }
            }
            if (!mbar_wait(act_bar, act_parity, b.err, abort_flag)) {
                drain(seq, qi, act_issued, act_parity);
                failed = true;
                break;
            }
            uint32_t xo = 0;
            int ubase = 0;
            for (int j = ja; j <= jb; j++) {
                if (!((act_mask >> j) & 1)) continue;
                const GemvJob& J = b.job[j];
                const float* xs = reinterpret_cast<const float*>(smem + b.off_x + xo);
                const int n_u = nt * J.units;
                for (int r = ((warp - ubase) % GV_WARPS + GV_WARPS) % GV_WARPS; r < n_u; r += GV_WARPS) {
                    float v[8];
                    unit_load(J, xs, r, lane, v);
                    unit_store(J, r, v, reinterpret_cast<int8_t*>(smem + J.act_q),
                               reinterpret_cast<float*>(smem + J.act_d), reinterpret_cast<int16_t*>(smem + J.act_s),
                               lane);
                }
                ubase += n_u;
                xo += (uint32_t)(nt * J.n_in * 4);
            }
            __syncthreads();
        } else {
        if (threadIdx.x == 0 && act_issued) {
            const int64_t nt = min((int64_t)NT, b.n_tok - t0);
            uint32_t tx = 0;
            for (int j = ja; j <= jb; j++) {
                if (!((act_mask >> j) & 1)) continue;
                const GemvJob& J = b.job[j];
                tx += (uint32_t)(nt * J.n_in + nt * J.ds * 4 + nt * sum_bytes(J.type, J.n_in));
            }
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(act_bar, tx);
            for (int j = ja; j <= jb; j++) {
                if (!((act_mask >> j) & 1)) continue;
                const GemvJob& J = b.job[j];
                // the converted activations of NT tokens fit where the layout put them
                // (a failed check leaves the phase short: the wait for it then runs out)
                if (!SYN_IN_BOUNDS((uint32_t)J.act_q + (uint32_t)(NT * J.n_in) <= dyn_smem_bytes() &&
                                   (uint32_t)J.act_d + (uint32_t)(NT * J.ds * 4) <= dyn_smem_bytes() &&
                                   (uint32_t)J.act_s + (uint32_t)(NT * sum_bytes(J.type, J.n_in)) <= dyn_smem_bytes()))
                    continue;
                bulk_g2s(smem_u32(smem + J.act_q), J.actg + t0 * J.n_in, (uint32_t)(nt * J.n_in), act_bar);
                bulk_g2s(smem_u32(smem + J.act_d), J.actg + J.g_d + t0 * J.ds * 4, (uint32_t)(nt * J.ds * 4), act_bar);
                if (J.type != SYN_Q8_0)
                    bulk_g2s(smem_u32(smem + J.act_s), J.actg + J.g_s + t0 * sum_bytes(J.type, J.n_in),
                             (uint32_t)(nt * sum_bytes(J.type, J.n_in)), act_bar);
            }
        }
        if (!mbar_wait(act_bar, act_parity, b.err, abort_flag)) {
            drain(seq, qi, act_issued, act_parity);
            failed = true;
            break;
        }
        }

        float acc[NT];
#pragma unroll
        for (int t = 0; t < NT; t++) acc[t] = 0.f;
        // packed rows: the window of steps whose row sums are reduced together
        constexpr int PW = Win<NT>::N;
        float part[PW][NT];
#pragma unroll
        for (int i = 0; i < PW; i++)
#pragma unroll
            for (int t = 0; t < NT; t++) part[i][t] = 0.f;
        int pw = 0;
        int64_t prow = r0;
        const int lgl = lg < 0 ? 0 : small_block(type) ? lg - 1 : lg + 1;  // log2 lanes per packed row
        const int rstep = lg < 0 ? 0 : bps >> lg;                          // packed rows per warp step
        int64_t crow = r0;
        int cbcol = b0;
        int cu = u0;
        uint32_t qc = seq;
        while (more(crow, cu)) {
            if (more(irow, iu)) {
                int nblk, nrows;
                extent(irow, ibcol, nblk, nrows);
                __syncwarp();
                issue(irow, ibcol, nblk, (qi++) % GV_NS);
                advance(irow, ibcol, nblk, nrows);
                iu++;
            }
            const uint32_t s = qc % GV_NS;
            if (!mbar_wait(bar0 + 8 * s, (qc / GV_NS) & 1, b.err, abort_flag)) {
                drain(qc, qi, false, 0);
                failed = true;
                break;
            }
            qc++;
            int nblk, nrows;
            extent(crow, cbcol, nblk, nrows);
            if (nblk <= 0) {  // cannot happen with a valid geometry; never spin without progress
                drain(qc, qi, false, 0);
                failed = true;
                break;
            }
            const uint8_t* sbase = ring + s * GV_SLOT + (int)(((crow * nb + cbcol) * (int64_t)bb) & 15);
            if (lg >= 0) {
                // rows of 2^lg <= bps blocks: rstep rows per warp step; the lanes of a row form
                // an aligned group of 2^lgl lanes.  Stages hold a multiple of rstep rows, so the
                // warp's steps cover its rows in order, rstep at a time.
                for (int s0 = 0; s0 < nblk; s0 += bps) {
                    lane_step<NT, FAM>(type, sbase, bb, s0, nblk - s0, s0, nb - 1, A, acc);
#pragma unroll
                    for (int i = 0; i + 1 < PW; i++)
#pragma unroll
                        for (int t = 0; t < NT; t++) part[i][t] = part[i + 1][t];
#pragma unroll
                    for (int t = 0; t < NT; t++) {
                        part[PW - 1][t] = acc[t];
                        acc[t] = 0.f;
                    }
                    if (++pw == PW) {
                        win_flush<NT>(part, PW, lgl, lane, prow, rstep, r1, Y, n_out, t0, b.n_tok);
                        prow += (int64_t)PW * rstep;
                        pw = 0;
                    }
                }
            } else {
                // wider rows: each row (or run of one row) takes ceil(blocks / bps) warp steps
                const int per_row = nrows > 0 ? nb : nblk;
                const int rows = nrows > 0 ? nrows : 1;
                const int bstart = nrows > 0 ? 0 : cbcol;
                for (int r = 0; r < rows; r++) {
                    const uint8_t* rowp = sbase + (int64_t)r * nb * bb;
                    for (int s0 = 0; s0 < per_row; s0 += bps)
                        lane_step<NT, FAM>(type, rowp, bb, s0, per_row - s0, bstart + s0, -1, A, acc);
                    if (nrows > 0 || split || cbcol + nblk == nb) {
#pragma unroll
                        for (int t = 0; t < NT; t++) {
                            const float v = warp_sum(acc[t]);
                            if (lane == 0 && t0 + t < b.n_tok && SYN_IN_BOUNDS(crow + r < n_out)) {
                                if (split) atomicAdd(Y + (t0 + t) * n_out + crow + r, v);
                                else Y[(t0 + t) * n_out + crow + r] = v;
                            }
                            acc[t] = 0.f;
                        }
                    }
                }
            }
            __syncwarp();
            advance(crow, cbcol, nblk, nrows);
            cu++;
        }
        if (!failed && pw > 0) win_flush<NT>(part, pw, lgl, lane, prow, rstep, r1, Y, n_out, t0, b.n_tok);
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
    const int64_t nbx = n_in / block_elems(type), ds = (nbx + 3) & ~int64_t(3);
    return n_in + ds * 4 + sum_bytes(type, n_in);
}

// Work partition of a launch: warps per matrix (and whether long rows are split into two
// runs), the warp -> matrix table, and whether the CTAs convert their own activations.
// x_need: the shared memory the fused conversion stages per CTA.
static cudaError_t plan_partition(GemvBatch& b, int sms, int NT, int64_t& x_need) {
    // Warps per matrix: the smallest per-warp byte bound T for which ceil(units / units per
    // warp) warps of every matrix fit in the grid (units per warp = floor(T / unit bytes)),
    // found by bisection; the warps left over go to the matrices in proportion to bytes.
    const int GW = sms * GV_WARPS;
    // cost of a unit: its bytes, weighted by the format's decode work per byte (percent)
    auto unit_bytes = [&](const GemvJob& J) {
        const int64_t by = J.upr > 1 ? (int64_t)J.stage_blocks * J.bb : J.row_bytes;
        const int64_t w = J.type == SYN_Q6_K ? SYN_GV_COST_Q6_K : J.type == SYN_Q8_0 ? SYN_GV_COST_Q8_0 : 100;
        return by * w / 100;
    };
    auto warps_for = [&](const GemvJob& J, int64_t T) {
        const int64_t per = std::max<int64_t>(1, T / unit_bytes(J));
        return (J.n_units + per - 1) / per;
    };
    auto bisect = [&]() {
        int64_t lo = 1, hi = 1;
        for (int j = 0; j < b.n_jobs; j++) hi = std::max<int64_t>(hi, (int64_t)b.job[j].n_units * unit_bytes(b.job[j]));
        while (lo < hi) {
            const int64_t T = lo + (hi - lo) / 2;
            int64_t need = 0;
            for (int j = 0; j < b.n_jobs; j++) need += warps_for(b.job[j], T);
            if (need <= GW) hi = T;
            else lo = T + 1;
        }
        return lo;
    };
    int64_t lo = bisect();
    // Rows of two stages are split into two runs only where that lowers the bound by more
    // than 5 %: whole rows need no zeroed Y and no atomic additions.
    bool any_split = false;
    for (int j = 0; j < b.n_jobs; j++) any_split |= b.job[j].upr > 1;
    if (any_split) {
        int upr_was[GEMV_MAX_JOBS];
        for (int j = 0; j < b.n_jobs; j++) {
            GemvJob& J = b.job[j];
            upr_was[j] = J.upr;
            J.upr = 1;
            J.n_units = (int)J.n_out;
        }
        const int64_t whole = bisect();
        if (whole * 100 > lo * 105) {
            for (int j = 0; j < b.n_jobs; j++) {
                GemvJob& J = b.job[j];
                J.upr = upr_was[j];
                J.n_units = (int)(J.n_out * J.upr);
            }
        } else {
            lo = whole;
        }
    }
    int64_t nw[GEMV_MAX_JOBS], used = 0;
    for (int j = 0; j < b.n_jobs; j++) {
        nw[j] = std::min<int64_t>(warps_for(b.job[j], lo), b.job[j].n_units);
        nw[j] = std::max<int64_t>(nw[j], 1);
        used += nw[j];
    }
    if (used > GW) return cudaErrorInvalidConfiguration;  // more matrices than warps
    const int64_t spare = GW - used;
    for (int j = 0; j < b.n_jobs && spare > 0; j++) {
        const GemvJob& J = b.job[j];
        const int64_t extra = (int64_t)((double)spare * (double)(J.n_out * J.row_bytes) / (double)b.total_bytes);
        nw[j] = std::min<int64_t>(nw[j] + extra, std::max<int64_t>(nw[j], J.n_units));
    }
    int w = 0;
    for (int j = 0; j < b.n_jobs; j++) {
        GemvJob& J = b.job[j];
        J.warp_begin = w;
        J.warp_end = w + (int)nw[j];
        for (int k = J.warp_begin; k < J.warp_end; k++) b.warp_job[k] = (uint8_t)j;
        w = J.warp_end;
    }
    for (int k = w; k < GW; k++) b.warp_job[k] = (uint8_t)(b.n_jobs - 1);  // idle: share of the last
    if (w < GW) b.job[b.n_jobs - 1].warp_end = GW;
    // the conversion kernel: a programmatic dependent of the preceding work on the stream
    // (it waits for that work to finish before touching memory); a previous decode launch
    // releases it early, so its launch latency overlaps that launch's tail
    for (int j = 0; j < b.n_jobs; j++) {
        GemvJob& J = b.job[j];
        J.units = small_block(J.type) ? (J.nbx + 3) / 4 : J.nbx;
    }
    // Each CTA converts the activations of its own matrices (staged in shared memory) when
    // that is at most one conversion unit per warp and the rows fit next to the rings: no
    // conversion launch and no workspace round trip.  More units per CTA cost more than the
    // launch they save (every CTA would repeat the divisions of the encoder).
    const int64_t nt = std::min<int64_t>(NT, b.n_tok);
    int64_t u_need = 0;
    x_need = 0;
    for (int c = 0; c < sms; c++) {
        int64_t xb = 0, ub = 0;
        const int ja = b.warp_job[c * GV_WARPS];
        b.act_mask[c] = 0;
        for (int j = ja; j <= b.warp_job[c * GV_WARPS + GV_WARPS - 1]; j++) {
            if (!first_reader(b, ja, j)) continue;
            b.act_mask[c] |= (uint16_t)(1u << j);
            xb += nt * b.job[j].n_in * 4;
            ub += nt * b.job[j].units;
        }
        x_need = std::max(x_need, xb);
        u_need = std::max(u_need, ub);
    }
    b.fused = u_need <= GV_WARPS && b.off_x + x_need <= 227 * 1024 ? 1 : 0;
    return cudaSuccess;
}

// The partition is a pure function of the shapes, and a decode loop repeats the same shapes
// every step; the bisection costs about as much host time as a launch, so the last few
// partitions are kept per host thread.
struct GemvPlanKey {
    int sms, n_jobs, nt_max, pad;
    int64_t n_tok;
    int type[GEMV_MAX_JOBS], upr[GEMV_MAX_JOBS], act_src[GEMV_MAX_JOBS];
    int64_t n_out[GEMV_MAX_JOBS], n_in[GEMV_MAX_JOBS];
};
struct GemvPlan {
    GemvPlanKey key;
    bool valid;
    int fused;
    int64_t x_need;
    int upr[GEMV_MAX_JOBS], n_units[GEMV_MAX_JOBS], warp_begin[GEMV_MAX_JOBS], warp_end[GEMV_MAX_JOBS];
    uint8_t warp_job[GV_MAX_SMS * GV_WARPS];
    uint16_t act_mask[GV_MAX_SMS];
};

static cudaError_t plan_cached(GemvBatch& b, int sms, int NT, int64_t& x_need) {
    static thread_local GemvPlan plans[4];
    static thread_local int next = 0;
    GemvPlanKey k;
    memset(&k, 0, sizeof(k));
    k.sms = sms;
    k.n_jobs = b.n_jobs;
    k.nt_max = NT;
    k.n_tok = b.n_tok;
    for (int j = 0; j < b.n_jobs; j++) {
        k.type[j] = b.job[j].type;
        k.upr[j] = b.job[j].upr;
        k.act_src[j] = b.job[j].act_src;
        k.n_out[j] = b.job[j].n_out;
        k.n_in[j] = b.job[j].n_in;
    }
    const int GW = sms * GV_WARPS;
    for (GemvPlan& P : plans) {
        if (!P.valid || memcmp(&P.key, &k, sizeof(k)) != 0) continue;
        for (int j = 0; j < b.n_jobs; j++) {
            GemvJob& J = b.job[j];
            J.upr = P.upr[j];
            J.n_units = P.n_units[j];
            J.warp_begin = P.warp_begin[j];
            J.warp_end = P.warp_end[j];
            J.units = small_block(J.type) ? (J.nbx + 3) / 4 : J.nbx;
        }
        memcpy(b.warp_job, P.warp_job, (size_t)GW);
        memcpy(b.act_mask, P.act_mask, sizeof(P.act_mask));
        b.fused = P.fused;
        x_need = P.x_need;
        return cudaSuccess;
    }
    const cudaError_t e = plan_partition(b, sms, NT, x_need);
    if (e != cudaSuccess) return e;
    GemvPlan& P = plans[next];
    next = (next + 1) % 4;
    P.key = k;
    for (int j = 0; j < b.n_jobs; j++) {
        P.upr[j] = b.job[j].upr;
        P.n_units[j] = b.job[j].n_units;
        P.warp_begin[j] = b.job[j].warp_begin;
        P.warp_end[j] = b.job[j].warp_end;
    }
    memcpy(P.warp_job, b.warp_job, (size_t)GW);
    memcpy(P.act_mask, b.act_mask, sizeof(P.act_mask));
    P.fused = b.fused;
    P.x_need = x_need;
    P.valid = true;
    return cudaSuccess;
}

template <int NT>
static cudaError_t run_gemv(GemvBatch& b, int sms, cudaStream_t s) {
    sms = std::min(sms, GV_MAX_SMS);  // one CTA per SM, up to the size of the warp table
    int64_t off = 0;
    for (int j = 0; j < b.n_jobs; j++) {
        GemvJob& J = b.job[j];
        if (J.act_src != j) {  // the shared input's area
            J.act_q = b.job[J.act_src].act_q;
            J.act_d = b.job[J.act_src].act_d;
            J.act_s = b.job[J.act_src].act_s;
            continue;
        }
        J.act_q = (int)off;
        off = up16(off + (int64_t)NT * J.n_in);
        J.act_d = (int)off;
        off = up16(off + (int64_t)NT * J.ds * 4);
        J.act_s = (int)off;
        off = up16(off + (int64_t)NT * sum_bytes(J.type, J.n_in));
    }
    off = (off + 127) & ~int64_t(127);
    b.off_stage = (int)off;
    off += (int64_t)GV_WARPS * GV_NS * GV_SLOT;
    b.off_bar = (int)off;
    off += GV_WARPS * GV_NS * 8;
    b.off_flag = (int)off;
    off += 16;  // abort flag, activation barrier
    if (off > 227 * 1024) return cudaErrorInvalidConfiguration;
    b.off_x = (int)up16(off);
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        void (*kerns[8])(GemvBatch) = {k_gemv<NT, false, 0>, k_gemv<NT, true, 0>, k_gemv<NT, false, 2>,
                                       k_gemv<NT, true, 2>,  k_gemv<NT, false, 3>, k_gemv<NT, true, 3>,
                                       k_gemv<NT, false, 4>, k_gemv<NT, true, 4>};
        for (auto k : kerns)
            if (attr_err == cudaSuccess)
                attr_err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    int64_t x_need = 0;
    const cudaError_t pe = plan_cached(b, sms, NT, x_need);
    if (pe != cudaSuccess) return pe;
    const size_t smem = b.fused ? (size_t)(b.off_x + x_need) : (size_t)b.off_x;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (b.fused) {
        // rows split between two warps are added into Y: zero it first
        for (int j = 0; j < b.n_jobs; j++) {
            const GemvJob& J = b.job[j];
            if (J.upr > 1) {
                const cudaError_t ez = cudaMemsetAsync(J.Y, 0, (size_t)(b.n_tok * J.n_out) * sizeof(float), s);
                if (ez != cudaSuccess) return ez;
            }
        }
    } else {
    // one row of 4-warp CTAs per matrix that converts its input or needs its Y zeroed, a warp
    // per unit (up to four SMs' worth of CTAs)
    int64_t max_units = 1, all_units = 0;
    b.n_conv = 0;
    for (int j = 0; j < b.n_jobs; j++) {
        const GemvJob& J = b.job[j];
        if (J.act_src == j) {
            max_units = std::max<int64_t>(max_units, b.n_tok * J.units);
            all_units += b.n_tok * J.units;
        }
        if (J.act_src == j || J.upr > 1) b.conv_job[b.n_conv++] = (uint8_t)j;
    }
    b.late_trigger = all_units >= GV_LATE_UNITS ? 1 : 0;
    const int64_t act_x = std::min<int64_t>((max_units + 3) / 4, std::max<int64_t>(1, (int64_t)sms * 4 / b.n_conv));
    cudaLaunchConfig_t acfg = {};
    acfg.gridDim = dim3((unsigned)act_x, (unsigned)b.n_conv);
    acfg.blockDim = dim3(128);
    acfg.stream = s;
    acfg.attrs = attr;
    acfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&acfg, k_act_decode, b);
    if (e != cudaSuccess) return e;
    }
    // the decode kernel, a programmatic dependent of the conversion launch (or, fused, of the
    // preceding work): it streams weights (which nothing before it writes) before it waits
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(GV_WARPS * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the instantiation for the launch's formats: all Q4_K, all Q6_K, all 32-weight, or mixed
    int fam = 0;
    if (SYN_GV_FAMILIES) {
        bool all_q4k = true, all_q6k = true, all_small = true;
        for (int j = 0; j < b.n_jobs; j++) {
            all_q4k = all_q4k && b.job[j].type == SYN_Q4_K;
            all_q6k = all_q6k && b.job[j].type == SYN_Q6_K;
            all_small = all_small && small_block(b.job[j].type);
        }
        fam = all_q4k ? 3 : all_q6k ? 4 : all_small ? 2 : 0;
    }
    if (fam == 3)
        return b.fused ? cudaLaunchKernelEx(&cfg, k_gemv<NT, true, 3>, b) : cudaLaunchKernelEx(&cfg, k_gemv<NT, false, 3>, b);
    if (fam == 4)
        return b.fused ? cudaLaunchKernelEx(&cfg, k_gemv<NT, true, 4>, b) : cudaLaunchKernelEx(&cfg, k_gemv<NT, false, 4>, b);
    if (fam == 2)
        return b.fused ? cudaLaunchKernelEx(&cfg, k_gemv<NT, true, 2>, b) : cudaLaunchKernelEx(&cfg, k_gemv<NT, false, 2>, b);
    return b.fused ? cudaLaunchKernelEx(&cfg, k_gemv<NT, true, 0>, b) : cudaLaunchKernelEx(&cfg, k_gemv<NT, false, 0>, b);
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
    J.nbx = (int)(d.n_in / block_elems(d.type));
    J.ds = (J.nbx + 3) & ~3;
    J.bps = small_block(d.type) ? 64 : 16;
    const int fit = GV_STAGE / J.bb;  // >= bps for every format (static_assert above)
    J.lg_nb = -1;
    const bool packed = J.nb <= J.bps && (J.nb & (J.nb - 1)) == 0 && !(small_block(d.type) && J.nb < 2);
    if (packed) {
        int lg = 0;
        while ((1 << lg) < J.nb) lg++;
        J.lg_nb = lg;
        J.stage_blocks = (fit / J.bps) * J.bps;  // whole rows, whole warp steps
    } else if (J.nb <= fit) {
        J.stage_blocks = (fit / J.nb) * J.nb;  // whole rows
    } else {
        J.stage_blocks = (fit / J.bps) * J.bps;  // runs of one row
    }
    J.upr = (J.nb > J.stage_blocks && J.nb <= 2 * J.stage_blocks) ? 2 : 1;
    J.n_units = (int)(d.n_out * J.upr);
}

int64_t gemv_act_bytes(int type, int64_t n_in) { return act_bytes_per_token(type, n_in) + 64; }

// Activation layouts: Q8_0 codes and scales; the same with block code sums (Q4_0, Q5_0);
// Q8_K codes, scales and 16-sums (the K-quants).  Products share a converted input only
// within one layout.
static int act_kind(int type) { return type == SYN_Q8_0 ? 0 : small_block(type) ? 1 : 2; }

// Global workspace of one matrix's converted activations (all tokens).
static int64_t act_global_bytes(int type, int64_t n_in, int64_t n_tok) {
    const int64_t nbx = n_in / block_elems(type), ds = (nbx + 3) & ~int64_t(3);
    return up16(n_tok * n_in) + up16(n_tok * ds * 4) + up16(n_tok * sum_bytes(type, n_in)) + 256;
}

int64_t gemv_workspace_bytes(int n, const GemvDesc* d, int64_t n_tok) {
    int64_t bytes = 0;
    for (int j = 0; j < n; j++) bytes += act_global_bytes(d[j].type, d[j].n_in, n_tok);
    return bytes + 256;
}

cudaError_t launch_gemv_batch(int n, const GemvDesc* d, int64_t n_tok, void* ws, int* err, int sms, bool no_split,
                              cudaStream_t s) {
    if (n < 1 || n > GEMV_MAX_JOBS) return cudaErrorInvalidValue;
    GemvBatch b{};
    b.n_jobs = n;
    b.n_tok = n_tok;
    b.err = err;
    int64_t bytes = 0, act = 0;
    uint8_t* g = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
    for (int j = 0; j < n; j++) {
        make_job(b.job[j], d[j], bytes);
        GemvJob& J = b.job[j];
        if (no_split) {
            J.upr = 1;
            J.n_units = (int)J.n_out;
        }
        bytes += d[j].n_out * b.job[j].row_bytes;
        // products that read the same input in the same activation layout share its conversion
        J.act_src = j;
        for (int i = 0; i < j; i++)
            if (d[i].X == d[j].X && d[i].n_in == d[j].n_in && act_kind(d[i].type) == act_kind(d[j].type)) {
                J.act_src = i;
                break;
            }
        if (J.act_src != j) {
            J.actg = b.job[J.act_src].actg;
            J.g_d = b.job[J.act_src].g_d;
            J.g_s = b.job[J.act_src].g_s;
            continue;
        }
        J.actg = g;
        J.g_d = up16(n_tok * J.n_in);
        J.g_s = J.g_d + up16(n_tok * J.ds * 4);
        g += (act_global_bytes(d[j].type, d[j].n_in, n_tok) + 255) & ~int64_t(255);
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


#ifdef SYN_DEBUG
SYN_BOUNDS_READER(debug_bounds_gemv)
#endif

}  // namespace syn

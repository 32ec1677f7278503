// gemm.cu — prefill product on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   Y[t][o] = sum_k W~[o][k] * x~[t][k]
//
// W~ is the weight block expanded to fp16 in shared memory (w = d*sc*q - dmin*m for Q4_K,
// d*sc*(q-32) for Q6_K, d*q for Q8_0: format table of "The GGML ecosystem, and where
// synapse fits", section 5) and x~ = fp16(d_x * q_x) is the activation after the
// conversion to the vec_dot_type ("Products: weights against quantized activations").
// The product of the quantized activations is what the pages define; only the fp16
// rounding of the two operands and the fp32 summation order differ from it.  Prefill is
// compute-bound at 2 * params * tokens FLOPs ("llama.cpp and GGUF", CPU and Edge
// Inference), so this path feeds the tensor cores.
//
// One persistent CTA per SM, warp-specialised, one 128 x BN output tile per work unit
// (BN <= 256 tokens), optionally split along K:
//   warp 0      producer: 1-D bulk copies of the raw weight super-blocks (128 rows x 256 k)
//               into a 2-deep raw ring; 2-D TMA loads of x~ tiles (BN x 64, 128-byte
//               swizzle) into a 3-deep operand ring;
//   warp 1      allocates 512 TMEM columns (two fp32 accumulators of 128 x 256) and issues
//               tcgen05.mma.cta_group::1.kind::f16 (M=128, N=BN, K=16) from one thread;
//   warps 2-9   dequantize: raw blocks -> fp16 A tile (128 x 64) in the canonical K-major
//               128-byte-swizzled layout the MMA descriptor reads;
//   warps 10-13 epilogue: tcgen05.ld 32x32b from TMEM, store (or add, when split) to Y.
// All hand-offs are mbarriers; every wait is bounded (clock64) and gives up with a
// recorded error instead of hanging.
#include <cuda.h>

#include <algorithm>

#include "kernels.h"
#include "quant_dev.cuh"

namespace syn {

constexpr int GEMM_BM = 128;
constexpr int GEMM_BK = 64;           // one 128-byte swizzle row of fp16
constexpr int GEMM_SUPER = 256;       // k per raw weight stage
constexpr int GEMM_STAGES = 3;        // operand ring depth
constexpr int GEMM_RAW_STAGES = 2;    // raw weight ring depth
constexpr int GEMM_THREADS = 14 * 32;
constexpr int GEMM_A_BYTES = GEMM_BM * GEMM_BK * 2;   // 16 KB
constexpr int GEMM_B_BYTES = 256 * GEMM_BK * 2;       // 32 KB (BN <= 256)

template <int T> struct GemmFmt;
// raw_row: bytes reserved per weight row in a raw stage (a 256-k slice plus the 16-byte
// alignment window); sb_bytes: bytes of that slice in memory.
template <> struct GemmFmt<SYN_Q4_K> { static constexpr int BB = 144, SB_BYTES = 144, RAW_ROW = 144 + 16; };
template <> struct GemmFmt<SYN_Q6_K> { static constexpr int BB = 210, SB_BYTES = 210, RAW_ROW = 240; };
template <> struct GemmFmt<SYN_Q8_0> { static constexpr int BB = 34, SB_BYTES = 272, RAW_ROW = 288; };

struct GemmParams {
    const uint8_t* W;
    float* Y;
    int* err;
    int64_t n_out, n_in, n_tok;
    int64_t row_bytes;
    int64_t total_floor16;
    int nb;          // weight blocks per row
    int n_super;     // 256-k super-steps per row (last one may be partial for Q8_0)
    int bn;          // tokens per tile (multiple of 16, <= 256)
    int n_m, n_n, n_split;
    int64_t n_units;
    int accumulate;  // 1: add into Y (split-K), 0: store
    uint32_t idesc;
};

// ---------------------------------------------------------------------------------------
// tcgen05 / TMA primitives (PTX ISA: tcgen05.alloc/mma/commit/ld, cp.async.bulk.tensor)
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), leading byte offset unused for this layout.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;             // leading byte offset 16 B (ignored)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset 1024 B
    d |= (uint64_t)1 << 46;             // descriptor version
    d |= (uint64_t)2 << 61;             // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

#define TMEM_LD32(taddr, r)                                                                            \
    asm volatile(                                                                                      \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"  \
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                      \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),            \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),        \
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),     \
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),     \
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])                                            \
        : "r"(taddr)                                                                                   \
        : "memory")

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 2^23 + b as a float for a byte b (selected from a word by __byte_perm): subtracting
// 2^23 afterwards gives b exactly, at full FP32 rate (no integer-to-float conversion).
__device__ __forceinline__ float byte_as_float_2p23(uint32_t word, int i) {
    return __int_as_float((int)__byte_perm(word, 0x4B000000u, 0x7440u | (uint32_t)i));
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------------------
// dequantize one thread's 32 consecutive k of one weight row into 16 packed halves
// ---------------------------------------------------------------------------------------

// Q4_K: 64-k step c of the super-block, half h (sub-block j = 2c + h).
__device__ __forceinline__ void deq32_q4_k(const uint8_t* blk, int c, int h, uint32_t out[16]) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const float D = h2f_bits(hdr.x & 0xFFFF), Dm = h2f_bits(hdr.x >> 16);
    const int j = 2 * c + h, jj = j & 3, sh = 8 * jj;
    int sc, mn;
    if (j < 4) {
        sc = (hdr.y >> sh) & 63;
        mn = (hdr.z >> sh) & 63;
    } else {
        sc = ((hdr.w >> sh) & 15) | (((hdr.y >> (sh + 6)) & 3) << 4);
        mn = ((hdr.w >> (sh + 4)) & 15) | (((hdr.z >> (sh + 6)) & 3) << 4);
    }
    const float S = D * (float)sc, M = Dm * (float)mn;
    const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c + 16);
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int w = 0; w < 8; w++) {
        const uint32_t v = (qw[w] >> (4 * h)) & 0x0F0F0F0Fu;
        float f[4];
#pragma unroll
        for (int i = 0; i < 4; i++) f[i] = fmaf(byte_as_float_2p23(v, i) - 8388608.0f, S, -M);
        out[2 * w] = pack_half2(f[0], f[1]);
        out[2 * w + 1] = pack_half2(f[2], f[3]);
    }
}

// Q6_K: 64-k step c of the super-block (half H = c/2), thread half h: quarter
// qd = 2*(c%2) + h of the half, weights l + 32*qd for l = 0..31.
__device__ __forceinline__ void deq32_q6_k(const uint8_t* blk, int c, int h, uint32_t out[16]) {
    const int H = c >> 1, qd = 2 * (c & 1) + h;
    const float D = h2f_bits(*reinterpret_cast<const uint16_t*>(blk + 208));
    const int8_t* scs = reinterpret_cast<const int8_t*>(blk + 192 + 8 * H + 2 * qd);
    const float S0 = D * (float)scs[0], S1 = D * (float)scs[1];
    const uint8_t* ql = blk + 64 * H + ((qd & 1) ? 32 : 0);
    const uint8_t* qh = blk + 128 + 32 * H;
    const int nsh = (qd >= 2) ? 4 : 0, hsh = 2 * qd;
#pragma unroll
    for (int w = 0; w < 8; w++) {
        const uint32_t lo = (lds_u32_any(ql + 4 * w) >> nsh) & 0x0F0F0F0Fu;
        const uint32_t hi = ((lds_u32_any(qh + 4 * w) >> hsh) & 0x03030303u) << 4;
        const uint32_t v = lo | hi;
        const float S = (w < 4) ? S0 : S1;
        float f[4];
#pragma unroll
        for (int i = 0; i < 4; i++) f[i] = (byte_as_float_2p23(v, i) - 8388640.0f) * S;
        out[2 * w] = pack_half2(f[0], f[1]);
        out[2 * w + 1] = pack_half2(f[2], f[3]);
    }
}

// Q8_0: one 34-byte block (32 k).
__device__ __forceinline__ void deq32_q8_0(const uint8_t* blk, uint32_t out[16]) {
    const float D = h2f_bits(*reinterpret_cast<const uint16_t*>(blk));
#pragma unroll
    for (int w = 0; w < 8; w++) {
        const uint32_t v = lds_u32_any(blk + 2 + 4 * w) ^ 0x80808080u;  // int8 -> offset binary
        float f[4];
#pragma unroll
        for (int i = 0; i < 4; i++) f[i] = (byte_as_float_2p23(v, i) - 8388736.0f) * D;
        out[2 * w] = pack_half2(f[0], f[1]);
        out[2 * w + 1] = pack_half2(f[2], f[3]);
    }
}

// ---------------------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------------------

struct GemmSmem {
    // offsets from the 1024-aligned dynamic shared-memory base
    static constexpr int A = 0;
    static constexpr int B = A + GEMM_STAGES * GEMM_A_BYTES;
    static constexpr int RAW = B + GEMM_STAGES * GEMM_B_BYTES;
};

template <int T>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap xmap, const GemmParams p) {
    using F = GemmFmt<T>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + GemmSmem::A;
    uint8_t* sB = smem + GemmSmem::B;
    uint8_t* sRaw = smem + GemmSmem::RAW;
    constexpr int RAW_STAGE = GEMM_BM * F::RAW_ROW;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRaw + GEMM_RAW_STAGES * RAW_STAGE);
    // barrier slots
    uint64_t* raw_full = bars;                              // [2]
    uint64_t* raw_empty = bars + 2;                         // [2]
    uint64_t* b_full = bars + 4;                            // [3]
    uint64_t* a_full = bars + 7;                            // [3]
    uint64_t* ab_empty = bars + 10;                         // [3]
    uint64_t* acc_full = bars + 13;                         // [2]
    uint64_t* acc_empty = bars + 15;                        // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 18);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            mbar_init(smem_u32(&raw_full[i]), 1);
            mbar_init(smem_u32(&raw_empty[i]), 8);
            mbar_init(smem_u32(&acc_full[i]), 1);
            mbar_init(smem_u32(&acc_empty[i]), 4);
        }
        for (int i = 0; i < GEMM_STAGES; i++) {
            mbar_init(smem_u32(&b_full[i]), 1);
            mbar_init(smem_u32(&a_full[i]), 8);
            mbar_init(smem_u32(&ab_empty[i]), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int64_t n_units = p.n_units;

    auto unit_coords = [&](int64_t u, int& m, int& n, int& ss0, int& ss1) {
        n = (int)(u % p.n_n);
        const int64_t rest = u / p.n_n;
        m = (int)(rest % p.n_m);
        const int ks = (int)(rest / p.n_m);
        ss0 = (int)((int64_t)ks * p.n_super / p.n_split);
        ss1 = (int)((int64_t)(ks + 1) * p.n_super / p.n_split);
    };
    // number of 64-k steps in super-step ss
    auto steps_in = [&](int ss) {
        const int64_t k0 = (int64_t)ss * GEMM_SUPER;
        const int64_t rem = p.n_in - k0;
        const int64_t st = (rem + GEMM_BK - 1) / GEMM_BK;
        return (int)(st < 4 ? st : 4);
    };

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        uint32_t rc = 0, kc = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            int m, n, ss0, ss1;
            unit_coords(u, m, n, ss0, ss1);
            for (int ss = ss0; ss < ss1 && ok; ss++) {
                const int rs = rc % GEMM_RAW_STAGES;
                if (!mbar_wait(smem_u32(&raw_empty[rs]), ((rc / GEMM_RAW_STAGES) & 1) ^ 1, p.err, abort_flag)) { ok = false; break; }
                // raw weight slice of 128 rows: per row one window-aligned bulk copy
                const int nblk_sb = (T == SYN_Q8_0) ? min(8, p.nb - ss * 8) : 1;
                const int64_t len = (int64_t)nblk_sb * F::BB;
                uint32_t my_tx = 0;
                int64_t a0[4], nbytes[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int r = lane + 32 * i;
                    const int64_t o = (int64_t)m * GEMM_BM + r;
                    a0[i] = 0; nbytes[i] = 0;
                    if (o < p.n_out) {
                        const int64_t src = o * p.row_bytes + (int64_t)ss * F::SB_BYTES;
                        const int64_t lo = src & ~int64_t(15);
                        int64_t hi = (src + len + 15) & ~int64_t(15);
                        if (hi > p.total_floor16) hi = p.total_floor16;
                        a0[i] = lo;
                        nbytes[i] = hi > lo ? hi - lo : 0;
                        my_tx += (uint32_t)nbytes[i];
                    }
                }
                uint8_t* rbase = sRaw + rs * RAW_STAGE;
                // The bytes of W past its last 16-byte boundary (end of the last row only),
                // by plain loads, before the arrive below publishes the stage.
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int r = lane + 32 * i;
                    const int64_t o = (int64_t)m * GEMM_BM + r;
                    if (o >= p.n_out) continue;
                    const int64_t src = o * p.row_bytes + (int64_t)ss * F::SB_BYTES;
                    const int64_t end = src + len;
                    if (end > p.total_floor16) {
                        const int64_t lo = src & ~int64_t(15);
                        for (int64_t k = (lo > p.total_floor16 ? lo : p.total_floor16); k < end; k++)
                            rbase[r * F::RAW_ROW + (k - lo)] = p.W[k];
                    }
                }
                uint32_t tx = my_tx;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tx += __shfl_xor_sync(0xffffffffu, tx, o);
                const uint32_t rfull = smem_u32(&raw_full[rs]);
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(rfull, tx);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; i++)
                    if (nbytes[i] > 0)
                        bulk_g2s(smem_u32(rbase + (lane + 32 * i) * F::RAW_ROW), p.W + a0[i], (uint32_t)nbytes[i], rfull);
                rc++;
                // activation tiles of this super-step
                const int nst = steps_in(ss);
                for (int k4 = 0; k4 < nst; k4++) {
                    const int ks = kc % GEMM_STAGES;
                    if (!mbar_wait(smem_u32(&ab_empty[ks]), ((kc / GEMM_STAGES) & 1) ^ 1, p.err, abort_flag)) { ok = false; break; }
                    if (lane == 0) {
                        const uint32_t bf = smem_u32(&b_full[ks]);
                        mbar_arrive_expect_tx(bf, (uint32_t)(p.bn * GEMM_BK * 2));
                        tma_load_2d(smem_u32(sB + ks * GEMM_B_BYTES), &xmap, ss * GEMM_SUPER + k4 * GEMM_BK,
                                    n * p.bn, bf);
                    }
                    __syncwarp();
                    kc++;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        uint32_t kc = 0, ac = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            int m, n, ss0, ss1;
            unit_coords(u, m, n, ss0, ss1);
            const int a = ac & 1;
            if (!mbar_wait(smem_u32(&acc_empty[a]), ((ac >> 1) & 1) ^ 1, p.err, abort_flag)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(a * 256);
            uint32_t first = 1;
            for (int ss = ss0; ss < ss1 && ok; ss++) {
                const int nst = steps_in(ss);
                for (int k4 = 0; k4 < nst; k4++) {
                    const int ks = kc % GEMM_STAGES;
                    const uint32_t par = (kc / GEMM_STAGES) & 1;
                    if (!mbar_wait(smem_u32(&a_full[ks]), par, p.err, abort_flag) ||
                        !mbar_wait(smem_u32(&b_full[ks]), par, p.err, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t a_addr = smem_u32(sA + ks * GEMM_A_BYTES);
                        const uint32_t b_addr = smem_u32(sB + ks * GEMM_B_BYTES);
#pragma unroll
                        for (int kk = 0; kk < GEMM_BK / 16; kk++) {
                            mma_f16(d_tmem, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(b_addr + kk * 32), p.idesc,
                                    first ? 0u : 1u);
                            first = 0;
                        }
                        mma_commit(smem_u32(&ab_empty[ks]));
                    }
                    __syncwarp();
                    kc++;
                }
            }
            if (!ok) break;
            if (lane == 0) mma_commit(smem_u32(&acc_full[a]));
            __syncwarp();
            ac++;
        }
    } else if (warp < 10) {
        // ------------------------------ dequantize ------------------------------
        const int dw = warp - 2;
        const int r = 32 * (dw & 3) + lane;   // row of the tile
        const int h = dw >> 2;                // k half of the 64-wide step
        uint32_t rc = 0, kc = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            int m, n, ss0, ss1;
            unit_coords(u, m, n, ss0, ss1);
            const int64_t o = (int64_t)m * GEMM_BM + r;
            const bool row_ok = o < p.n_out;
            for (int ss = ss0; ss < ss1 && ok; ss++) {
                const int rs = rc % GEMM_RAW_STAGES;
                if (!mbar_wait(smem_u32(&raw_full[rs]), (rc / GEMM_RAW_STAGES) & 1, p.err, abort_flag)) { ok = false; break; }
                const int64_t src = o * p.row_bytes + (int64_t)ss * F::SB_BYTES;
                const uint8_t* row = sRaw + rs * RAW_STAGE + r * F::RAW_ROW + (int)(src & 15);
                const int nst = steps_in(ss);
                for (int k4 = 0; k4 < nst; k4++) {
                    const int ks = kc % GEMM_STAGES;
                    if (!mbar_wait(smem_u32(&ab_empty[ks]), ((kc / GEMM_STAGES) & 1) ^ 1, p.err, abort_flag)) { ok = false; break; }
                    uint32_t out[16];
                    const int64_t kglob = (int64_t)ss * GEMM_SUPER + k4 * GEMM_BK + h * 32;
                    if (row_ok && kglob < p.n_in) {
                        if (T == SYN_Q4_K) deq32_q4_k(row, k4, h, out);
                        else if (T == SYN_Q6_K) deq32_q6_k(row, k4, h, out);
                        else deq32_q8_0(row + (2 * k4 + h) * 34, out);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; i++) out[i] = 0u;
                    }
                    // 128-byte swizzle: 16-byte chunk j of row r lands at chunk j ^ (r % 8)
                    uint8_t* arow = sA + ks * GEMM_A_BYTES + r * 128;
#pragma unroll
                    for (int cidx = 0; cidx < 4; cidx++) {
                        const int j = 4 * h + cidx;
                        *reinterpret_cast<uint4*>(arow + ((j ^ (r & 7)) << 4)) =
                            make_uint4(out[4 * cidx], out[4 * cidx + 1], out[4 * cidx + 2], out[4 * cidx + 3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&a_full[ks]));
                    kc++;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&raw_empty[rs]));
                rc++;
            }
        }
    } else {
        // ------------------------------ epilogue ------------------------------
        const int quarter = warp & 3;
        uint32_t ac = 0;
        for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
            int m, n, ss0, ss1;
            unit_coords(u, m, n, ss0, ss1);
            const int a = ac & 1;
            if (!mbar_wait(smem_u32(&acc_full[a]), (ac >> 1) & 1, p.err, abort_flag)) break;
            tc_fence_after();
            const int64_t o = (int64_t)m * GEMM_BM + 32 * quarter + lane;
            const int64_t t0 = (int64_t)n * p.bn;
            for (int cb = 0; cb < p.bn; cb += 32) {
                uint32_t v[32];
                const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(a * 256 + cb);
                TMEM_LD32(taddr, v);
                tmem_ld_wait();
                if (o < p.n_out) {
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        const int64_t t = t0 + cb + i;
                        if (cb + i < p.bn && t < p.n_tok) {
                            float* dst = p.Y + t * p.n_out + o;
                            if (p.accumulate) atomicAdd(dst, __uint_as_float(v[i]));
                            else *dst = __uint_as_float(v[i]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[a]));
            ac++;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled get_encode() {
    static PFN_encodeTiled fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_encodeTiled>(ptr);
    }
    return fn;
}

static size_t gemm_smem_bytes(int raw_row) {
    return 1024 /* alignment slack */ + GemmSmem::RAW + (size_t)GEMM_RAW_STAGES * GEMM_BM * raw_row + 256;
}

// Pick the K split so that units fill the SMs in whole waves: minimise
// ceil(tiles * S / sms) / S, preferring the smaller S on ties (each split keeps >= 2
// super-steps).
static int pick_split(int64_t tiles, int n_super, int sms) {
    int best = 1;
    double best_t = 1e30;
    for (int S = 1; S <= 16; S++) {
        if (S > 1 && n_super / S < 2) break;
        const int64_t waves = (tiles * S + sms - 1) / sms;
        const double t = (double)waves / S + (S > 1 ? 0.02 : 0.0);
        if (t < best_t - 1e-9) {
            best_t = t;
            best = S;
        }
    }
    return best;
}

template <int T>
static cudaError_t run_gemm(GemmParams p, const CUtensorMap& map, int sms, cudaStream_t s) {
    using F = GemmFmt<T>;
    const size_t smem = gemm_smem_bytes(F::RAW_ROW);
    auto kern = k_gemm<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(p.n_units, sms);
    kern<<<(unsigned)grid, GEMM_THREADS, smem, s>>>(map, p);
    return cudaGetLastError();
}

cudaError_t launch_gemm(int type, const void* W, int64_t n_out, int64_t n_in, const void* xh, int64_t n_tok,
                        float* Y, int* err, int sms, cudaStream_t s) {
    PFN_encodeTiled encode = get_encode();
    if (!encode) return cudaErrorNotSupported;
    GemmParams p{};
    p.W = static_cast<const uint8_t*>(W);
    p.Y = Y;
    p.err = err;
    p.n_out = n_out;
    p.n_in = n_in;
    p.n_tok = n_tok;
    p.nb = (int)(n_in / block_elems(type));
    p.row_bytes = (int64_t)p.nb * block_bytes(type);
    p.total_floor16 = (n_out * p.row_bytes) & ~int64_t(15);
    p.n_super = (int)((n_in + GEMM_SUPER - 1) / GEMM_SUPER);
    p.bn = (int)std::min<int64_t>(256, (n_tok + 15) / 16 * 16);
    p.n_m = (int)((n_out + GEMM_BM - 1) / GEMM_BM);
    p.n_n = (int)((n_tok + p.bn - 1) / p.bn);
    p.n_split = pick_split((int64_t)p.n_m * p.n_n, p.n_super, sms);
    p.n_units = (int64_t)p.n_m * p.n_n * p.n_split;
    p.accumulate = p.n_split > 1 ? 1 : 0;
    // kind::f16 instruction descriptor: D fp32, A and B fp16, both K-major, N, M = 128
    p.idesc = (1u << 4) | ((uint32_t)(p.bn >> 3) << 17) | ((uint32_t)(GEMM_BM >> 4) << 24);

    CUtensorMap map;
    cuuint64_t dims[2] = {(cuuint64_t)n_in, (cuuint64_t)n_tok};
    cuuint64_t strides[1] = {(cuuint64_t)n_in * 2};
    cuuint32_t box[2] = {(cuuint32_t)GEMM_BK, (cuuint32_t)p.bn};
    cuuint32_t estr[2] = {1, 1};
    CUresult cr = encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(xh), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (p.accumulate) {
        cudaError_t e = cudaMemsetAsync(Y, 0, (size_t)n_tok * n_out * sizeof(float), s);
        if (e != cudaSuccess) return e;
    }
    switch (type) {
    case SYN_Q4_K: return run_gemm<SYN_Q4_K>(p, map, sms, s);
    case SYN_Q6_K: return run_gemm<SYN_Q6_K>(p, map, sms, s);
    case SYN_Q8_0: return run_gemm<SYN_Q8_0>(p, map, sms, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace syn

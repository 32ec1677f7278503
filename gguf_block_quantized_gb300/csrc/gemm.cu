// gemm.cu — prefill product on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   Y[t][o] = sum_k W~[o][k] * x~[t][k]
//
// W~ is the weight block expanded to fp16 in shared memory (w = d*sc*q - dmin*m for Q4_K,
// d*sc*(q-32) for Q6_K, d*q for Q8_0: format table of "The GGML ecosystem, and where
// synapse fits", section 5) and x~ = fp16(d_x * q_x) is the activation after the
// conversion to the vec_dot_type ("Products: weights against quantized activations").
// The product of the quantized activations is what the pages define; only the fp16
// rounding of the operands (and of the sub-block scales) and the fp32 summation order
// differ from it.  Prefill is compute-bound at 2 * params * tokens FLOPs ("llama.cpp and
// GGUF", CPU and Edge Inference), so this path feeds the tensor cores.
//
// One persistent CTA per SM, warp-specialised, one 128 x BN output tile per work unit
// (BN <= 256 tokens).  Tiles that do not fill the SMs in whole waves are split along K (all
// of them, or only those of the last, partial wave; a cost model picks): the units of a
// split tile add their partial sums into a Y zeroed beforehand.  Warp roles (mapped to
// warps by kGemmRoles in the dequantizing kernels, so as to keep the MMA issuer's
// sub-partition clear of dequantizers):
//   role 0      raw-weight producer: 128 rows x 256 k of weight blocks per raw stage, by
//               one 2-D TMA load when the row pitch is a multiple of 16 bytes (else one
//               1-D bulk copy per row);
//   role 1      allocates 512 TMEM columns (two fp32 accumulators of 128 x 256) and issues
//               tcgen05.mma.cta_group::1.kind::f16 (M=128, N=BN, K=16) from one thread;
//   role 2      activation producer: 2-D TMA loads of x~ tiles (BN x 64, 128-byte swizzle)
//               into a 3-deep operand ring (it alone waits for the conversion kernel);
//   roles 3-18  dequantize, two teams of 8 taking alternate 64-k steps: raw blocks -> fp16
//               A tile (128 x 64) in the canonical K-major 128-byte-swizzled layout the MMA
//               descriptor reads, in half2 arithmetic (F16 weights: no dequantization, role 0
//               loads the fp16 tile by TMA straight into that layout);
//   roles 19-22 epilogue: tcgen05.ld 32x32b from TMEM, then per warp a 32 x 16 staging box
//               and one 2-D TMA store (or reduce-add, when split along K) to Y.
// All hand-offs are mbarriers; every wait is bounded (clock64) and gives up with a
// recorded error instead of hanging.  Index arithmetic is 32-bit: 64-bit division runs on
// the fp64 pipe.
#include <cuda.h>

#include <algorithm>
#include <climits>
#include <cmath>

#include "kernels.h"
#include "quant_dev.cuh"

namespace syn {

constexpr int GEMM_BM = 128;
constexpr int GEMM_BK = 64;           // one 128-byte swizzle row of fp16
constexpr int GEMM_SUPER = 256;       // k per raw weight stage
// dequantizer teams: team t handles the 64-k steps with step index = t (mod teams); each
// team is 8 warps (128 rows x two 32-k halves)
#ifndef SYN_GEMM_DEQ_TEAMS
#define SYN_GEMM_DEQ_TEAMS 2
#endif
constexpr int GEMM_DEQ_TEAMS = SYN_GEMM_DEQ_TEAMS;
constexpr int GEMM_DEQ_WARP0 = 3, GEMM_DEQ_WARPS = 8 * GEMM_DEQ_TEAMS, GEMM_EPI_WARP0 = 3 + GEMM_DEQ_WARPS;
// Warp roles, numbered: 0 raw-weight producer, 1 MMA issuer (and TMEM owner), 2 activation
// producer, 3 .. 3 + GEMM_DEQ_WARPS - 1 dequantizers, then the 4 epilogue warps.  A warp runs
// on sub-partition (warp index % 4), and an epilogue warp reads only the TMEM lanes of its own
// sub-partition, so the four epilogue warps sit on four different ones.  Dequantizing
// kernels run 24 warps laid out by kGemmRoles so that the MMA warp's sub-partition holds one
// dequantizer instead of four: they otherwise take most of its issue slots and the MMAs go
// out late (measured, Q4_K: FFN up at 512 tokens 64.7 -> 58.8 us, FFN down at 2048 tokens
// 235.6 -> 210.1 us).  The fp16-weight kernel (no dequantizers) keeps 23 warps in role order
// (the table's layout measured 4-8 % slower for it).
constexpr int GEMM_ROLE_IDLE = 31;
static_assert(GEMM_DEQ_WARPS == 16, "the role table is laid out for two teams of 8 dequantizers");
__constant__ uint8_t kGemmRoles[24] = {GEMM_EPI_WARP0, 1, GEMM_EPI_WARP0 + 1, GEMM_EPI_WARP0 + 2, 3, 0, 4, 5, 6, 2,
                                       7, 8, 9, GEMM_EPI_WARP0 + 3, 10, 11, 12, 13, 14, 15, 16, GEMM_ROLE_IDLE, 17,
                                       18};
template <int T>
constexpr int gemm_warps() {
    return T == SYN_F16 ? GEMM_EPI_WARP0 + 4 : 24;
}
constexpr int GEMM_A_BYTES = GEMM_BM * GEMM_BK * 2;   // 16 KB
constexpr int GEMM_B_BYTES = 256 * GEMM_BK * 2;       // 32 KB (BN <= 256)
constexpr int GEMM_OUT_TOK = 16;                      // tokens per output staging chunk
constexpr int GEMM_OUT_BYTES = GEMM_BM * GEMM_OUT_TOK * 4;  // four warps x 32 outputs x 16 tokens, fp32

template <int T> struct GemmFmt;
// SB_BYTES: bytes of a 256-k slice of one row; BOX: bytes per row of the 2-D TMA box that
// covers the slice from the 16-byte boundary at or below it (ESIZE: the tensor map's
// element size, 2 where the box is wider than 256 elements of one byte); RAW_ROW: bytes
// reserved per row in a raw stage for the per-row copy windows; RAW_STAGES: ring depth.
// A_STAGES / B_STAGES: depths of the dequantized-weight and activation rings, measured per
// format: a deeper A ring (5 stages) lets the two dequantizer teams run ahead of the MMA,
// and 2-3 activation stages cover the L2 latency of the activation tiles.
#ifndef SYN_GEMM_Q4K_RAW
#define SYN_GEMM_Q4K_RAW 2
#endif
#ifndef SYN_GEMM_Q4K_A
#define SYN_GEMM_Q4K_A 5
#endif
#ifndef SYN_GEMM_Q4K_B
#define SYN_GEMM_Q4K_B 3
#endif
template <int R, int A, int B> struct GemmDepth {
    static constexpr int RAW_STAGES = R, A_STAGES = A, B_STAGES = B;
};
template <> struct GemmFmt<SYN_Q4_K> : GemmDepth<SYN_GEMM_Q4K_RAW, SYN_GEMM_Q4K_A, SYN_GEMM_Q4K_B> {
    static constexpr int BB = 144, SB_BYTES = 144, BOX = 144, ESIZE = 1, RAW_ROW = 144;
};
#ifndef SYN_GEMM_Q6K_RAW
#define SYN_GEMM_Q6K_RAW 2
#endif
#ifndef SYN_GEMM_Q6K_A
#define SYN_GEMM_Q6K_A 5
#endif
#ifndef SYN_GEMM_Q6K_B
#define SYN_GEMM_Q6K_B 2
#endif
template <> struct GemmFmt<SYN_Q6_K> : GemmDepth<SYN_GEMM_Q6K_RAW, SYN_GEMM_Q6K_A, SYN_GEMM_Q6K_B> {
    static constexpr int BB = 210, SB_BYTES = 210, BOX = 240, ESIZE = 1, RAW_ROW = 240;
};
// ring depths (raw, A, B) of the other formats
#ifndef SYN_GEMM_Q40_A
#define SYN_GEMM_Q40_A 5
#endif
#ifndef SYN_GEMM_Q40_B
#define SYN_GEMM_Q40_B 3
#endif
#ifndef SYN_GEMM_Q50_A
#define SYN_GEMM_Q50_A 3
#endif
#ifndef SYN_GEMM_Q50_B
#define SYN_GEMM_Q50_B 3
#endif
#ifndef SYN_GEMM_F16_A
#define SYN_GEMM_F16_A 4
#endif
#ifndef SYN_GEMM_F16_B
#define SYN_GEMM_F16_B 4
#endif
#ifndef SYN_GEMM_Q80_A
#define SYN_GEMM_Q80_A 3
#endif
#ifndef SYN_GEMM_Q80_B
#define SYN_GEMM_Q80_B 3
#endif
template <> struct GemmFmt<SYN_Q4_0> : GemmDepth<2, SYN_GEMM_Q40_A, SYN_GEMM_Q40_B> {
    static constexpr int BB = 18, SB_BYTES = 144, BOX = 144, ESIZE = 1, RAW_ROW = 160;
};
template <> struct GemmFmt<SYN_Q5_0> : GemmDepth<2, SYN_GEMM_Q50_A, SYN_GEMM_Q50_B> {
    static constexpr int BB = 22, SB_BYTES = 176, BOX = 176, ESIZE = 1, RAW_ROW = 192;
};
// F16: no raw ring; the weight tile is loaded by TMA straight into the A ring (the same
// 128-byte-swizzled K-major layout as the activation tiles)
template <> struct GemmFmt<SYN_F16> : GemmDepth<1, SYN_GEMM_F16_A, SYN_GEMM_F16_B> {  // (one raw stage of 0 bytes: unused)
    static constexpr int BB = 2, SB_BYTES = 512, BOX = 128, ESIZE = 2, RAW_ROW = 0;
};
template <> struct GemmFmt<SYN_Q8_0> : GemmDepth<2, SYN_GEMM_Q80_A, SYN_GEMM_Q80_B> {
    static constexpr int BB = 34, SB_BYTES = 272, BOX = 272, ESIZE = 2, RAW_ROW = 288;
};

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
    int m_full;      // m-tiles [0, m_full) run whole (one unit each, stored); the others are
                     // split n_split ways along K (their units add into a zeroed Y)
    int u_full;      // m_full * n_n: units of whole tiles, numbered first
    int n_units;
    int accumulate;  // 1: some units add into Y (split-K)
    int raw_tma;     // 1: weight slices by one 2-D TMA load per stage (row_bytes % 16 == 0)
    int raw_row;     // bytes per row in a raw stage: BOX (TMA) or RAW_ROW (per-row copies)
    int y_tma;       // 1: Y written by 2-D TMA stores / reduce-adds (n_out % 4 == 0)
    int streamk_work;  // > 0: stream-K schedule: tiles [0, sk_tile0) whole, round robin, then
                       // the tiles x super-steps of tiles [sk_tile0, n_m * n_n) (this many,
                       // < 2^31) dealt to the CTAs in equal contiguous ranges, each range cut
                       // at tile boundaries into units; a unit that is not a whole tile adds
                       // into Y (zeroed first).  0: the units below, round robin
    int sk_tile0;      // stream-K: the first tile of the shared range (a multiple of n_n)
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

// shared -> global 2-D tile store and reduce-add (fp32 add, performed at L2), bulk-group
// completion
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
                 "r"(c0), "r"(c1), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, int c0, int c1, uint32_t src) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
                 "r"(c0), "r"(c1), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

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

// ---------------------------------------------------------------------------------------
// dequantize one thread's 32 consecutive k of one weight row into 16 packed halves, in
// half2 arithmetic: a byte b becomes the fp16 1024 + b by a byte permute with 0x64 (the
// upper byte of 1024.0) and the offset is subtracted exactly.  The sub-block scale S = d*sc
// and min M = dmin*m are exact in fp32 but not in fp16; rounding them would bias every
// weight of the sub-block the same way (for Q4_K the q*S and M terms nearly cancel, so a
// relative 2^-12 on either is a large error on w).  They are therefore split into a head
// and a tail scaled by 2^12 (both normal fp16 numbers, together exact):
//     w = fp16( (q*S_hi - M_hi) + 2^-12 * (q*S_lo' - M_lo') )
// three fma per pair of weights, each rounding relative to |w|, not to |S| or |M|.
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// v (exact in fp32) -> head fp16(v) and tail fp16((v - head) * 2^12), both broadcast
__device__ __forceinline__ void split_h2(float v, __half2& hi, __half2& lo) {
    const __half h = __float2half_rn(v);
    hi = __half2half2(h);
    lo = __float2half2_rn((v - __half2float(h)) * 4096.0f);
}

// bytes (b0, b1) of v -> half2(1024 + b0, 1024 + b1); bytes (b2, b3) likewise
__device__ __forceinline__ __half2 bytes01_h2(uint32_t v) { return u32_as_h2(__byte_perm(v, 0x64646464u, 0x4140)); }
__device__ __forceinline__ __half2 bytes23_h2(uint32_t v) { return u32_as_h2(__byte_perm(v, 0x64646464u, 0x4342)); }

// The scales a dequantizing thread needs in one 256-k super-step are decoded once, when the
// raw stage arrives: a thread expands row r, k-half h of the two 64-k steps c0 and c0 + 2 of
// the super-step that its team takes (c0 = 0 or 1).

// Q4_K: the thread's sub-blocks are j = 2c + h: j0 = 2*c0 + h (scales in the low words)
// and j0 + 4 (high words).  The 1024 of the byte permute is folded into the offset:
// w = S*(1024 + q) - (1024*S + M).
struct Q4Prep {
    __half2 Sh[2], Sl[2], nCh[2], nCl[2];
};
__device__ __forceinline__ void prep_q4_k(const uint8_t* blk, int c0, int h, Q4Prep& P) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const float D = h2f_bits(hdr.x & 0xFFFF), Dm = h2f_bits(hdr.x >> 16);
    // 6-bit scales / mins of sub-blocks 0..3 and 4..7, one per byte
    const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, mn_lo = hdr.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t mn_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    const uint32_t sel = 0x4440u | (uint32_t)(2 * c0 + h);
    const float S0 = D * (float)__byte_perm(sc_lo, 0, sel), M0 = Dm * (float)__byte_perm(mn_lo, 0, sel);
    const float S1 = D * (float)__byte_perm(sc_hi, 0, sel), M1 = Dm * (float)__byte_perm(mn_hi, 0, sel);
    split_h2(S0, P.Sh[0], P.Sl[0]);
    split_h2(-fmaf(1024.0f, S0, M0), P.nCh[0], P.nCl[0]);
    split_h2(S1, P.Sh[1], P.Sl[1]);
    split_h2(-fmaf(1024.0f, S1, M1), P.nCh[1], P.nCl[1]);
}
// step c = c0 + 2i of the super-block
__device__ __forceinline__ void deq32_q4_k(const uint8_t* blk, int c, int h, const Q4Prep& P, int i, uint32_t out[16]) {
    const __half2 tail = __float2half2_rn(1.0f / 4096.0f);
    // (selects, not indexing: a runtime index would put the struct in local memory)
    const __half2 Sh = i ? P.Sh[1] : P.Sh[0], Sl = i ? P.Sl[1] : P.Sl[0];
    const __half2 nCh = i ? P.nCh[1] : P.nCh[0], nCl = i ? P.nCl[1] : P.nCl[0];
    const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c + 16);
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int w = 0; w < 8; w++) {
        const uint32_t v = (qw[w] >> (4 * h)) & 0x0F0F0F0Fu;
        const __half2 qa = bytes01_h2(v), qb = bytes23_h2(v);
        out[2 * w] = h2_as_u32(__hfma2(__hfma2(qa, Sl, nCl), tail, __hfma2(qa, Sh, nCh)));
        out[2 * w + 1] = h2_as_u32(__hfma2(__hfma2(qb, Sl, nCl), tail, __hfma2(qb, Sh, nCh)));
    }
}

// Q6_K: step c covers half H = c / 2 of the block; the thread expands quarter
// qd = 2*(c % 2) + h of that half (weights l + 32*qd, l = 0..31, sub-blocks 2*qd and
// 2*qd + 1 of the half).  For steps c0 and c0 + 2: qd = 2*c0 + h in halves 0 and 1.
struct Q6Prep {
    __half2 Sh[2][2], Sl[2][2];
};
__device__ __forceinline__ void prep_q6_k(const uint8_t* blk, int c0, int h, Q6Prep& P) {
    const float D = h2f_bits(*reinterpret_cast<const uint16_t*>(blk + 208));
    const int8_t* scs = reinterpret_cast<const int8_t*>(blk + 192);
    const int qd = 2 * c0 + h;
    const int s00 = scs[2 * qd], s01 = scs[2 * qd + 1], s10 = scs[8 + 2 * qd], s11 = scs[9 + 2 * qd];
    split_h2(D * (float)s00, P.Sh[0][0], P.Sl[0][0]);
    split_h2(D * (float)s01, P.Sh[0][1], P.Sl[0][1]);
    split_h2(D * (float)s10, P.Sh[1][0], P.Sl[1][0]);
    split_h2(D * (float)s11, P.Sh[1][1], P.Sl[1][1]);
}
__device__ __forceinline__ void deq32_q6_k(const uint8_t* blk, int c, int h, const Q6Prep& P, int i, uint32_t out[16]) {
    const int H = c >> 1, qd = 2 * (c & 1) + h;
    const __half2 k1056 = __float2half2_rn(1056.0f);  // 1024 + 32
    const __half2 tail = __float2half2_rn(1.0f / 4096.0f);
    uint32_t ql[8], qh[8];
    lds_words_any<8>(blk + 64 * H + ((qd & 1) ? 32 : 0), ql);
    lds_words_any<8>(blk + 128 + 32 * H, qh);
    const int nsh = (qd >= 2) ? 4 : 0, hsh = 2 * qd;
    const __half2 S0h = i ? P.Sh[1][0] : P.Sh[0][0], S0l = i ? P.Sl[1][0] : P.Sl[0][0];
    const __half2 S1h = i ? P.Sh[1][1] : P.Sh[0][1], S1l = i ? P.Sl[1][1] : P.Sl[0][1];
#pragma unroll
    for (int w = 0; w < 8; w++) {
        const uint32_t lo = (ql[w] >> nsh) & 0x0F0F0F0Fu;
        const uint32_t hi = ((qh[w] >> hsh) & 0x03030303u) << 4;
        const uint32_t v = lo | hi;
        const __half2 Sh = (w < 4) ? S0h : S1h, Sl = (w < 4) ? S0l : S1l;
        const __half2 qa = __hsub2(bytes01_h2(v), k1056), qb = __hsub2(bytes23_h2(v), k1056);
        out[2 * w] = h2_as_u32(__hfma2(__hmul2(qa, Sl), tail, __hmul2(qa, Sh)));
        out[2 * w + 1] = h2_as_u32(__hfma2(__hmul2(qb, Sl), tail, __hmul2(qb, Sh)));
    }
}

// Q8_0: one 34-byte block (32 k).  The scale is stored in fp16, so one rounding of q*D.
__device__ __forceinline__ void deq32_q8_0(const uint8_t* blk, uint32_t out[16]) {
    const __half2 D = u32_as_h2(__byte_perm(*reinterpret_cast<const uint16_t*>(blk), 0, 0x1010));
    const __half2 k1152 = __float2half2_rn(1152.0f);  // 1024 + 128
    uint32_t q[8];
    lds_words_any<8>(blk + 2, q);
#pragma unroll
    for (int w = 0; w < 8; w++) {
        const uint32_t v = q[w] ^ 0x80808080u;  // int8 -> offset binary
        out[2 * w] = h2_as_u32(__hmul2(__hsub2(bytes01_h2(v), k1152), D));
        out[2 * w + 1] = h2_as_u32(__hmul2(__hsub2(bytes23_h2(v), k1152), D));
    }
}

// Q4_0 / Q5_0 (OFF = 8 / 16): one 18- / 22-byte block (32 k), codes q[l] / q[l + 16] in the
// low / high nibble of byte l (Q5_0: fifth bits in a 32-bit word before them); w = D*(q - OFF)
// with D stored in fp16: one rounding.
template <int OFF>
__device__ __forceinline__ void deq32_qx_0(const uint8_t* blk, uint32_t out[16]) {
    const __half2 D = u32_as_h2(__byte_perm(*reinterpret_cast<const uint16_t*>(blk), 0, 0x1010));
    const __half2 kOff = __float2half2_rn(1024.0f + OFF);
    uint32_t w[5];
    if (OFF == 8) lds_words_any<4>(blk + 2, w + 1);
    else lds_words_any<5>(blk + 2, w);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint32_t lo = w[1 + i] & 0x0F0F0F0Fu, hi = (w[1 + i] >> 4) & 0x0F0F0F0Fu;
        if (OFF == 16) {
            lo |= ((((w[0] >> (4 * i)) & 15u) * 0x00204081u) & 0x01010101u) << 4;
            hi |= ((((w[0] >> (16 + 4 * i)) & 15u) * 0x00204081u) & 0x01010101u) << 4;
        }
        out[2 * i] = h2_as_u32(__hmul2(__hsub2(bytes01_h2(lo), kOff), D));
        out[2 * i + 1] = h2_as_u32(__hmul2(__hsub2(bytes23_h2(lo), kOff), D));
        out[8 + 2 * i] = h2_as_u32(__hmul2(__hsub2(bytes01_h2(hi), kOff), D));
        out[8 + 2 * i + 1] = h2_as_u32(__hmul2(__hsub2(bytes23_h2(hi), kOff), D));
    }
}

// ---------------------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------------------

template <int T>
struct GemmSmem {
    // offsets from the 1024-aligned dynamic shared-memory base
    static constexpr int A = 0;
    static constexpr int B = A + GemmFmt<T>::A_STAGES * GEMM_A_BYTES;
    static constexpr int RAW = B + GemmFmt<T>::B_STAGES * GEMM_B_BYTES;
    static constexpr int OUT = RAW + GemmFmt<T>::RAW_STAGES * GEMM_BM * GemmFmt<T>::RAW_ROW;
    static constexpr int BARS = OUT + GEMM_OUT_BYTES;
};

// unit u -> tile (m, n) and k range [ss0, ss1) in 256-k super-steps (32-bit arithmetic)
__device__ __forceinline__ void unit_coords(const GemmParams& p, int u, int& m, int& n, int& ss0, int& ss1,
                                            bool& add) {
    if (u < p.u_full) {  // a whole tile
        m = u / p.n_n;
        n = u - m * p.n_n;
        ss0 = 0;
        ss1 = p.n_super;
        add = false;
        return;
    }
    const int v = u - p.u_full, ts = p.n_m - p.m_full;
    const int rest = v / p.n_n;
    n = v - rest * p.n_n;
    const int ks = rest / ts;
    m = p.m_full + (rest - ks * ts);
    ss0 = (ks * p.n_super) / p.n_split;
    ss1 = ((ks + 1) * p.n_super) / p.n_split;
    add = p.n_split > 1;
}
__device__ __forceinline__ void unit_coords(const GemmParams& p, int u, int& m, int& n, int& ss0, int& ss1) {
    bool add;
    unit_coords(p, u, m, n, ss0, ss1, add);
}

// The units of this CTA, in order (every role of the CTA walks the same sequence): round
// robin over the unit list, or (stream-K) round robin over the whole tiles before sk_tile0,
// then the CTA's range of the shared tile x super-step work.
struct UnitIter {
    int u;      // round robin: the next unit (stream-K: the next whole tile)
    int g, g1;  // stream-K: the next and the end of this CTA's tile x super-step range
    __device__ explicit UnitIter(const GemmParams& p) {
        u = blockIdx.x;
        const int g0 = p.sk_tile0 * p.n_super;
        g = g0 + (int)(((int64_t)p.streamk_work * blockIdx.x) / gridDim.x);
        g1 = g0 + (int)(((int64_t)p.streamk_work * (blockIdx.x + 1)) / gridDim.x);
    }
    __device__ void stop(const GemmParams& p) {
        u = INT_MAX;
        g = g1;
    }
    __device__ bool next(const GemmParams& p, int& m, int& n, int& ss0, int& ss1, bool& add) {
        if (p.streamk_work > 0) {
            if (u < p.sk_tile0) {  // a whole tile of the leading full waves
                m = u / p.n_n;
                n = u - m * p.n_n;
                ss0 = 0;
                ss1 = p.n_super;
                add = false;
                u += (int)gridDim.x;
                return true;
            }
            if (g >= g1) return false;
            const int t = g / p.n_super;  // tile: m-major, its token tiles next to each other
            ss0 = g - t * p.n_super;
            const int end = min(g1, (t + 1) * p.n_super);
            ss1 = end - t * p.n_super;
            m = t / p.n_n;
            n = t - m * p.n_n;
            add = !(ss0 == 0 && ss1 == p.n_super);
            g = end;
            return true;
        }
        if (u >= p.n_units) return false;
        unit_coords(p, u, m, n, ss0, ss1, add);
        u += (int)gridDim.x;
        return true;
    }
};

template <int T>
__global__ void __launch_bounds__(32 * gemm_warps<T>(), 1)
    k_gemm(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
           const __grid_constant__ CUtensorMap ymap, const GemmParams p) {
    using F = GemmFmt<T>;
    using L = GemmSmem<T>;
    constexpr int RS = F::RAW_STAGES;
    constexpr int GEMM_A_STAGES = F::A_STAGES;
    constexpr int GEMM_B_STAGES = F::B_STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + L::A;
    uint8_t* sB = smem + L::B;
    uint8_t* sRaw = smem + L::RAW;
    constexpr int RAW_STAGE = GEMM_BM * F::RAW_ROW;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BARS);
    uint64_t* raw_full = bars;                              // [RS]
    uint64_t* raw_empty = bars + RS;                        // [RS]
    uint64_t* b_full = bars + 2 * RS;                       // [B stages]
    uint64_t* b_empty = b_full + GEMM_B_STAGES;             // [B stages] (MMA done with B stage)
    uint64_t* a_full = b_empty + GEMM_B_STAGES;             // [A stages]
    uint64_t* a_empty = a_full + GEMM_A_STAGES;             // [A stages] (MMA done with A stage)
    uint64_t* acc_full = a_empty + GEMM_A_STAGES;           // [2]
    uint64_t* acc_empty = acc_full + 2;                     // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(acc_empty + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int role = T == SYN_F16 ? warp : (int)kGemmRoles[warp];

    if (threadIdx.x == 0) {
        for (int i = 0; i < RS; i++) {
            mbar_init(smem_u32(&raw_full[i]), 1);
            mbar_init(smem_u32(&raw_empty[i]), GEMM_DEQ_WARPS);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(smem_u32(&acc_full[i]), 1);
            mbar_init(smem_u32(&acc_empty[i]), 4);
        }
        for (int i = 0; i < GEMM_B_STAGES; i++) {
            mbar_init(smem_u32(&b_full[i]), 1);
            mbar_init(smem_u32(&b_empty[i]), 1);
        }
        for (int i = 0; i < GEMM_A_STAGES; i++) {
            mbar_init(smem_u32(&a_full[i]), T == SYN_F16 ? 1 : 8);
            mbar_init(smem_u32(&a_empty[i]), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // number of 64-k steps in super-step ss
    auto steps_in = [&](int ss) {
        const int64_t rem = p.n_in - (int64_t)ss * GEMM_SUPER;
        const int64_t st = (rem + GEMM_BK - 1) / GEMM_BK;
        return (int)(st < 4 ? st : 4);
    };

    if (role == 0 && T == SYN_F16) {
        // ------------------------------ F16 weight tiles ------------------------------
        // 2-D TMA of 128 rows x 64 k of fp16 straight into the A ring (zero fill past
        // n_out / n_in)
        uint32_t kc = 0;
        bool ok = true;
        UnitIter it(p);
        int m, n, ss0, ss1;
        bool add;
        while (ok && it.next(p, m, n, ss0, ss1, add)) {
            for (int ss = ss0; ss < ss1 && ok; ss++) {
                const int nst = steps_in(ss);
                for (int k4 = 0; k4 < nst; k4++, kc++) {
                    const int ka = kc % GEMM_A_STAGES;
                    if (!mbar_wait(smem_u32(&a_empty[ka]), ((kc / GEMM_A_STAGES) & 1) ^ 1, p.err, abort_flag)) { ok = false; break; }
                    if (lane == 0) {
                        const uint32_t af = smem_u32(&a_full[ka]);
                        const int x = ss * GEMM_SUPER + k4 * GEMM_BK;
                        // a tile of this unit, its x on a 16-byte boundary (TMA)
                        const bool in = SYN_IN_BOUNDS(m * GEMM_BM < p.n_out && x < p.n_in && (x * 2) % 16 == 0);
                        mbar_arrive_expect_tx(af, in ? (uint32_t)GEMM_A_BYTES : 0u);
                        if (in) tma_load_2d(smem_u32(sA + ka * GEMM_A_BYTES), &wmap, x, m * GEMM_BM, af);
                    }
                    __syncwarp();
                }
            }
        }
        // the tiles still in flight (issued, not consumed: only after an abort) land first
        for (uint32_t i = kc > (uint32_t)GEMM_A_STAGES ? kc - GEMM_A_STAGES : 0u; i < kc; i++)
            mbar_drain(smem_u32(&a_full[i % GEMM_A_STAGES]), (i / GEMM_A_STAGES) & 1, p.err);
    } else if (role == 0) {
        // ------------------------------ raw weight producer ------------------------------
        uint32_t rc = 0;
        UnitIter it(p);
        int m, n, ss0, ss1;
        bool add;
        while (it.next(p, m, n, ss0, ss1, add)) {
            bool ok = true;
            for (int ss = ss0; ss < ss1; ss++) {
                const int rs = rc % RS;
                if (!mbar_wait(smem_u32(&raw_empty[rs]), ((rc / RS) & 1) ^ 1, p.err, abort_flag)) { ok = false; break; }
                if (p.raw_tma) {
                    // the whole 128-row slice in one load; rows past n_out and bytes past the
                    // row end are filled with zeros (and counted in the transaction bytes)
                    if (lane == 0) {
                        const uint32_t rfull = smem_u32(&raw_full[rs]);
                        const int x = (int)((((int64_t)ss * F::SB_BYTES) & ~int64_t(15)) / F::ESIZE);
                        // the slice lies in the box (from its 16-byte boundary), x is aligned,
                        // the tile starts inside W
                        const bool in = SYN_IN_BOUNDS(
                            (int)(((int64_t)ss * F::SB_BYTES) & 15) + F::SB_BYTES <= p.raw_row &&
                            (x * F::ESIZE) % 16 == 0 && (int64_t)m * GEMM_BM < p.n_out && ss < p.n_super);
                        mbar_arrive_expect_tx(rfull, in ? (uint32_t)(GEMM_BM * F::BOX) : 0u);
                        if (in) tma_load_2d(smem_u32(sRaw + rs * RAW_STAGE), &wmap, x, m * GEMM_BM, rfull);
                    }
                    __syncwarp();
                    rc++;
                    continue;
                }
                // raw weight slice of 128 rows: per row one window-aligned bulk copy
                const int nblk_sb = small_block(T) ? min(8, p.nb - ss * 8) : 1;
                const int64_t len = (int64_t)nblk_sb * F::BB;
                uint32_t my_tx = 0;
                int64_t a0[4];
                uint32_t nbytes[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int r = lane + 32 * i;
                    const int64_t o = (int64_t)m * GEMM_BM + r;
                    a0[i] = 0;
                    nbytes[i] = 0;
                    if (o < p.n_out) {
                        const int64_t src = o * p.row_bytes + (int64_t)ss * F::SB_BYTES;
                        const int64_t lo = src & ~int64_t(15);
                        int64_t hi = (src + len + 15) & ~int64_t(15);
                        if (hi > p.total_floor16) hi = p.total_floor16;
                        a0[i] = lo;
                        nbytes[i] = hi > lo ? (uint32_t)(hi - lo) : 0u;
                        // the window fits the row's space in the stage and lies inside W
                        if (!SYN_IN_BOUNDS(nbytes[i] <= (uint32_t)p.raw_row && lo >= 0 && hi <= p.total_floor16))
                            nbytes[i] = 0;
                        my_tx += nbytes[i];
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
                            if (SYN_IN_BOUNDS(k - lo < p.raw_row && k < p.n_out * p.row_bytes))
                                rbase[r * p.raw_row + (k - lo)] = p.W[k];
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
                        bulk_g2s(smem_u32(rbase + (lane + 32 * i) * p.raw_row), p.W + a0[i], nbytes[i], rfull);
                rc++;
            }
            if (!ok) break;
        }
        // the slices still in flight (issued, not consumed: only after an abort) land first
        for (uint32_t i = rc > (uint32_t)RS ? rc - RS : 0u; i < rc; i++)
            mbar_drain(smem_u32(&raw_full[i % RS]), (i / RS) & 1, p.err);
    } else if (role == 2) {
        // ------------------------------ activation producer ------------------------------
        // x~ is written by the conversion kernel this launch may overlap with: wait for it
        asm volatile("griddepcontrol.wait;" ::: "memory");
        uint32_t kc = 0;
        UnitIter it(p);
#ifdef SYN_TEST_STALL
        it.stop(p);  // timeout-test build: no activation tile is ever loaded, so the waits for one run out
#endif
        int m, n, ss0, ss1;
        bool add;
        while (it.next(p, m, n, ss0, ss1, add)) {
            bool ok = true;
            for (int ss = ss0; ss < ss1 && ok; ss++) {
                const int nst = steps_in(ss);
                for (int k4 = 0; k4 < nst; k4++) {
                    const int ks = kc % GEMM_B_STAGES;
                    if (!mbar_wait(smem_u32(&b_empty[ks]), ((kc / GEMM_B_STAGES) & 1) ^ 1, p.err, abort_flag)) { ok = false; break; }
                    if (lane == 0) {
                        const uint32_t bf = smem_u32(&b_full[ks]);
                        const int x = ss * GEMM_SUPER + k4 * GEMM_BK;
                        const bool in = SYN_IN_BOUNDS((int64_t)n * p.bn < p.n_tok && x < p.n_in && (x * 2) % 16 == 0 &&
                                                      p.bn * GEMM_BK * 2 <= GEMM_B_BYTES);
                        mbar_arrive_expect_tx(bf, in ? (uint32_t)(p.bn * GEMM_BK * 2) : 0u);
                        if (in) tma_load_2d(smem_u32(sB + ks * GEMM_B_BYTES), &xmap, x, n * p.bn, bf);
                    }
                    __syncwarp();
                    kc++;
                }
            }
            if (!ok) break;
        }
        // the tiles still in flight (issued, not consumed: only after an abort) land first
        for (uint32_t i = kc > (uint32_t)GEMM_B_STAGES ? kc - GEMM_B_STAGES : 0u; i < kc; i++)
            mbar_drain(smem_u32(&b_full[i % GEMM_B_STAGES]), (i / GEMM_B_STAGES) & 1, p.err);
    } else if (role == 1) {
        // ------------------------------ MMA issuer ------------------------------
        uint32_t kc = 0, ac = 0;
        bool ok = true;
        UnitIter it(p);
        int m, n, ss0, ss1;
        bool add;
        while (ok && it.next(p, m, n, ss0, ss1, add)) {
            // the unit is a tile of the product and a non-empty range of its K steps
            (void)SYN_IN_BOUNDS(m >= 0 && m < p.n_m && n >= 0 && n < p.n_n && ss0 >= 0 && ss0 < ss1 &&
                                ss1 <= p.n_super);
            const int a = ac & 1;
            if (!mbar_wait(smem_u32(&acc_empty[a]), ((ac >> 1) & 1) ^ 1, p.err, abort_flag)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(a * 256);
            uint32_t first = 1;
            for (int ss = ss0; ss < ss1 && ok; ss++) {
                const int nst = steps_in(ss);
                for (int k4 = 0; k4 < nst; k4++) {
                    const int ka = kc % GEMM_A_STAGES, kb = kc % GEMM_B_STAGES;
                    if (!mbar_wait(smem_u32(&a_full[ka]), (kc / GEMM_A_STAGES) & 1, p.err, abort_flag) ||
                        !mbar_wait(smem_u32(&b_full[kb]), (kc / GEMM_B_STAGES) & 1, p.err, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t a_addr = smem_u32(sA + ka * GEMM_A_BYTES);
                        const uint32_t b_addr = smem_u32(sB + kb * GEMM_B_BYTES);
#pragma unroll
                        for (int kk = 0; kk < GEMM_BK / 16; kk++) {
                            mma_f16(d_tmem, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(b_addr + kk * 32), p.idesc,
                                    first ? 0u : 1u);
                            first = 0;
                        }
                        mma_commit(smem_u32(&a_empty[ka]));
                        mma_commit(smem_u32(&b_empty[kb]));
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
        // every MMA issued has finished reading shared memory and writing TMEM before the
        // accumulators are freed (the commit of the last A stage tracks all earlier MMAs;
        // on the normal path the epilogue has already seen them finish)
        if (kc > 0)
            mbar_drain(smem_u32(&a_empty[(kc - 1) % GEMM_A_STAGES]), ((kc - 1) / GEMM_A_STAGES) & 1, p.err);
    } else if (role < GEMM_EPI_WARP0) {
      if (T != SYN_F16) {  // F16: no dequantization, the weights arrive as fp16
        // ------------------------------ dequantize ------------------------------
        const int dw = role - GEMM_DEQ_WARP0;
        const int r = 32 * (dw & 3) + lane;   // row of the tile
        const int h = (dw >> 2) & 1;          // k half of the 64-wide step
        const uint32_t team = (uint32_t)(dw >> 3);
        uint32_t rc = 0, kc = 0;
        bool ok = true;
        UnitIter it(p);
        int m, n, ss0, ss1;
        bool add;
        while (ok && it.next(p, m, n, ss0, ss1, add)) {
            const int64_t o = (int64_t)m * GEMM_BM + r;
            const bool row_ok = o < p.n_out;
            for (int ss = ss0; ss < ss1 && ok; ss++) {
                const int rs = rc % RS;
                if (!mbar_wait(smem_u32(&raw_full[rs]), (rc / RS) & 1, p.err, abort_flag)) { ok = false; break; }
                const int64_t src = o * p.row_bytes + (int64_t)ss * F::SB_BYTES;
                const uint8_t* row = sRaw + rs * RAW_STAGE + r * p.raw_row + (int)(src & 15);
                const int nst = steps_in(ss);
                // the slice read below lies in this row's space of the stage
                const bool row_in = SYN_IN_BOUNDS((int)(src & 15) + F::SB_BYTES <= p.raw_row);
                // this team's steps of the super-step: c0 and c0 + 2 (K-quants: 4 steps each)
                const int c0 = (int)((team + GEMM_DEQ_TEAMS - kc % GEMM_DEQ_TEAMS) % GEMM_DEQ_TEAMS);
                Q4Prep p4;
                Q6Prep p6;
                if (T == SYN_Q4_K && row_ok && row_in) prep_q4_k(row, c0, h, p4);
                if (T == SYN_Q6_K && row_ok && row_in) prep_q6_k(row, c0, h, p6);
                for (int k4 = 0; k4 < nst; k4++, kc++) {
                    if (kc % GEMM_DEQ_TEAMS != team) continue;
                    const int ks = kc % GEMM_A_STAGES;
                    uint32_t out[16];
                    const int64_t kglob = (int64_t)ss * GEMM_SUPER + k4 * GEMM_BK + h * 32;
                    if (row_ok && row_in && kglob < p.n_in) {
                        if (T == SYN_Q4_K) deq32_q4_k(row, k4, h, p4, k4 >> 1, out);
                        else if (T == SYN_Q6_K) deq32_q6_k(row, k4, h, p6, k4 >> 1, out);
                        else if (T == SYN_Q8_0) deq32_q8_0(row + (2 * k4 + h) * 34, out);
                        else deq32_qx_0<T == SYN_Q4_0 ? 8 : 16>(row + (2 * k4 + h) * F::BB, out);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; i++) out[i] = 0u;
                    }
                    if (!mbar_wait(smem_u32(&a_empty[ks]), ((kc / GEMM_A_STAGES) & 1) ^ 1, p.err, abort_flag)) { ok = false; break; }
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
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&raw_empty[rs]));
                rc++;
            }
        }
      }
    } else if (role != GEMM_ROLE_IDLE) {
        // ------------------------------ epilogue ------------------------------
        // TMEM -> registers (32 columns per load); then either through a per-warp staging
        // buffer of 32 outputs x 16 tokens and one 2-D TMA store (or reduce-add, for split
        // products) per buffer, clipped by the tensor map at n_out / n_tok, the four warps
        // independent of each other, or (rows whose pitch is not a multiple of 16 bytes)
        // per-element stores / atomic adds.
        const int quarter = warp & 3;
        float* stage = reinterpret_cast<float*>(smem + L::OUT + quarter * (GEMM_OUT_BYTES / 4));
        const uint32_t stage_s = smem_u32(stage);
        uint32_t ac = 0;
        UnitIter it(p);
        int m, n, ss0, ss1;
        bool add;
        while (it.next(p, m, n, ss0, ss1, add)) {
            const int a = ac & 1;
            if (!mbar_wait(smem_u32(&acc_full[a]), (ac >> 1) & 1, p.err, abort_flag)) break;
            tc_fence_after();
            const int o0 = m * GEMM_BM + 32 * quarter;
            const int64_t o = (int64_t)o0 + lane;
            const int t0 = n * p.bn;
            for (int cb = 0; cb < p.bn; cb += 32) {
                uint32_t v[32];
                const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(a * 256 + cb);
                TMEM_LD32(taddr, v);
                tmem_ld_wait();
                if (cb + 32 >= p.bn) {
                    // the accumulator is in registers: hand it back to the MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&acc_empty[a]));
                }
                if (p.y_tma) {
#pragma unroll
                    for (int hh = 0; hh < 2; hh++) {
                        const int tt = t0 + cb + GEMM_OUT_TOK * hh;
                        if (cb + GEMM_OUT_TOK * hh >= p.bn || tt >= p.n_tok || o0 >= p.n_out) continue;
                        if (lane == 0) bulk_wait_read<0>();  // the previous buffer has left the stage
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < GEMM_OUT_TOK; i++) stage[i * 32 + lane] = __uint_as_float(v[GEMM_OUT_TOK * hh + i]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            // x of the store on a 16-byte boundary, never negative
                            if (SYN_IN_BOUNDS(o0 >= 0 && (o0 * 4) % 16 == 0 && tt >= 0)) {
                                if (add) tma_reduce_add_2d(&ymap, o0, tt, stage_s);
                                else tma_store_2d(&ymap, o0, tt, stage_s);
                            }
                            bulk_commit();
                        }
                    }
                } else if (o < p.n_out) {
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        const int64_t t = (int64_t)t0 + cb + i;
                        if (cb + i < p.bn && t < p.n_tok && SYN_IN_BOUNDS(t * p.n_out + o < p.n_tok * p.n_out)) {
                            float* dst = p.Y + t * p.n_out + o;
                            if (add) atomicAdd(dst, __uint_as_float(v[i]));
                            else *dst = __uint_as_float(v[i]);
                        }
                    }
                }
            }
            ac++;
        }
        if (lane == 0) bulk_wait_all();  // Y written before the CTA (and its staging) goes away
        __syncwarp();
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
    // looked up once (a function-local static is initialised once, whatever the threads)
    static const PFN_encodeTiled fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_encodeTiled>(ptr);
        return static_cast<PFN_encodeTiled>(nullptr);
    }();
    return fn;
}

template <int T>
constexpr size_t gemm_smem_bytes() {
    return 1024 /* alignment slack */ + GemmSmem<T>::BARS + 256 /* barriers, TMEM slot, abort flag */;
}
static_assert(gemm_smem_bytes<SYN_Q4_K>() <= 232448 && gemm_smem_bytes<SYN_Q6_K>() <= 232448 &&
                  gemm_smem_bytes<SYN_Q8_0>() <= 232448 && gemm_smem_bytes<SYN_Q4_0>() <= 232448 &&
                  gemm_smem_bytes<SYN_Q5_0>() <= 232448 && gemm_smem_bytes<SYN_F16>() <= 232448,
              "shared memory per CTA exceeds 227 KB");
template <int T>
constexpr bool gemm_bars_fit() {
    return 8 * (2 * GemmFmt<T>::RAW_STAGES + 2 * GemmFmt<T>::A_STAGES + 2 * GemmFmt<T>::B_STAGES + 4) + 16 <= 256;
}
static_assert(gemm_bars_fit<SYN_Q4_K>() && gemm_bars_fit<SYN_Q6_K>() && gemm_bars_fit<SYN_Q8_0>() &&
                  gemm_bars_fit<SYN_Q4_0>() && gemm_bars_fit<SYN_Q5_0>() && gemm_bars_fit<SYN_F16>(),
              "barrier area");

// Cost model of a K split (microseconds on GB300, fitted to measured Q4_K products): whole
// waves of units, each 1/S of a tile's multiply-adds at about 7 TFLOP/s per SM plus a fixed
// pipeline cost; for S > 1, zeroing Y and adding S partial tiles into it at L2.
#ifndef SYN_GEMM_SM_TFLOPS
#define SYN_GEMM_SM_TFLOPS 7.0
#endif
#ifndef SYN_GEMM_UNIT_US
#define SYN_GEMM_UNIT_US 1.0
#endif
#ifndef SYN_GEMM_ZERO_US_PER_MB
#define SYN_GEMM_ZERO_US_PER_MB 0.15
#endif
#ifndef SYN_GEMM_ADD_US_PER_MB
#define SYN_GEMM_ADD_US_PER_MB 0.08
#endif

struct SplitPlan {
    int S;       // K split of the split tiles (1: none)
    int m_full;  // m-tiles run whole; the rest are split S ways (stream-K: shared)
    bool streamk = false;  // instead: the stream-K schedule (the whole tiles of m-tiles below
                           // m_full, then every CTA the same number of super-steps of the
                           // rest), where the cost model prefers it
};

#ifndef SYN_GEMM_STREAMK
#define SYN_GEMM_STREAMK 1
#endif
#ifndef SYN_GEMM_SK_TAIL
#define SYN_GEMM_SK_TAIL 1
#endif

// Pick the schedule of least modelled time, the smaller S on ties: S = 1 (whole tiles), every
// tile split S ways, or whole tiles for the full waves and only the m-tiles of the last,
// partial wave split S ways (their Y columns are then the only ones zeroed and added into).
// Each split keeps >= 2 super-steps.
static SplitPlan pick_split(int n_m, int n_n, int n_super, int sms, int bn, int64_t n_out, int64_t n_tok) {
    const int64_t tiles = (int64_t)n_m * n_n;
    const double tile_us = 2.0 * GEMM_BM * bn * (double)n_super * GEMM_SUPER / (SYN_GEMM_SM_TFLOPS * 1e6);
    auto y_mb = [&](int m_full) {
        const int64_t cols = n_out - (int64_t)m_full * GEMM_BM;
        return cols > 0 ? 4.0 * (double)cols * (double)n_tok / 1e6 : 0.0;
    };
    // m-tiles whose every token tile fits in the full waves
    const int m_tail_from = (int)std::min<int64_t>(n_m, (tiles / sms) * sms / n_n);
    SplitPlan best{1, n_m};
    double best_t = (double)((tiles + sms - 1) / sms) * (tile_us + SYN_GEMM_UNIT_US);
    for (int S = 2; S <= 16; S++) {
        if (n_super / S < 2) break;
        const double add = SYN_GEMM_ZERO_US_PER_MB + S * SYN_GEMM_ADD_US_PER_MB;
        for (int m_full : {0, m_tail_from}) {
            if (m_full >= n_m) continue;
            const int64_t u_full = (int64_t)m_full * n_n, u_tail = (tiles - u_full) * S;
            const double t = (double)((u_full + sms - 1) / sms) * (tile_us + SYN_GEMM_UNIT_US) +
                             (double)((u_tail + sms - 1) / sms) * (tile_us / S + SYN_GEMM_UNIT_US) + y_mb(m_full) * add;
            if (t < best_t * (1.0 - 1e-9)) {
                best_t = t;
                best = SplitPlan{S, m_full};
            }
            if (m_tail_from == 0) break;  // the two schedules coincide
        }
    }
    // stream-K: every CTA the same number of super-steps (cut into units at tile boundaries),
    // the Y columns of the shared tiles zeroed, and about two partial tiles per CTA added into
    // them.  Over all tiles it was measured faster only where the tiles do not fill one wave
    // and K is long (Q4_K FFN down at 512 tokens: 74.6 -> 72.5 us), slower for products of
    // short K or several waves (q/k/o at 512 and 2048 tokens +1.7 to +2.5 us, Q6_K FFN down at
    // 2048 tokens +4.4 us).  Where the tiles fill at least one wave, only the tiles of the last,
    // partial wave are shared (the full waves run whole tiles, as above): Q4_K FFN down at 2048
    // tokens 244.8 -> 235.8 us, Q6_K 281.5 -> 279.0; for K of 16 super-steps (q/o at 2048
    // tokens, the lm_head) it lost to the split tail by ~1 %, so it too needs long K.
    auto streamk_us = [&](int m_full) {
        const int64_t dp = (int64_t)m_full * n_n, shared = tiles - dp;
        const double W = (double)shared * n_super;
        const double t_ss = tile_us / n_super;
        const double partial = std::min((double)shared + sms, 2.0 * sms);
        const double tile_mb = 4.0 * GEMM_BM * bn / 1e6;
        return (double)((dp + sms - 1) / sms) * (tile_us + SYN_GEMM_UNIT_US) + std::ceil(W / sms) * t_ss +
               ((double)shared / sms + 1.0) * SYN_GEMM_UNIT_US + y_mb(m_full) * SYN_GEMM_ZERO_US_PER_MB +
               partial * tile_mb * SYN_GEMM_ADD_US_PER_MB;
    };
    if (SYN_GEMM_STREAMK && tiles * n_super < (int64_t(1) << 30)) {
        int m_sk = -1;
        if (tiles < sms && n_super >= 32) m_sk = 0;
        else if (SYN_GEMM_SK_TAIL && tiles >= sms && n_super >= 32 && m_tail_from > 0 && m_tail_from < n_m)
            m_sk = m_tail_from;
        if (m_sk >= 0 && streamk_us(m_sk) < best_t * (1.0 - 1e-9)) {
            best = SplitPlan{1, m_sk};
            best.streamk = true;
        }
    }
    return best;
}

template <int T>
static cudaError_t run_gemm(GemmParams p, const CUtensorMap& map, const CUtensorMap& wmap, const CUtensorMap& ymap,
                           int sms, cudaStream_t s) {
    const size_t smem = gemm_smem_bytes<T>();
    auto kern = k_gemm<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = std::min(p.n_units, sms);
    // launched as the programmatic dependent of the activation conversion: the weight
    // producer and the dequantizers start before the conversion has finished
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * gemm_warps<T>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, map, wmap, ymap, p);
}

static int gemm_bn(int64_t n_tok) { return (int)std::min<int64_t>(256, (n_tok + 15) / 16 * 16); }

static SplitPlan plan_of(int64_t n_out, int64_t n_in, int64_t n_tok, int sms) {
    const int bn = gemm_bn(n_tok);
    const int n_m = (int)((n_out + GEMM_BM - 1) / GEMM_BM), n_n = (int)((n_tok + bn - 1) / bn);
    const int n_super = (int)((n_in + GEMM_SUPER - 1) / GEMM_SUPER);
    return pick_split(n_m, n_n, n_super, sms, bn, n_out, n_tok);
}

// The schedule the prefill product takes (host only): out[0] = S (K split of the split
// tiles, 1: none), out[1] = m_full (row tiles run whole), out[2] = 1 for stream-K (the tiles of
// row tiles >= m_full shared), out[3] = the number of tiles.
void gemm_plan(int64_t n_out, int64_t n_in, int64_t n_tok, int sms, int out[4]) {
    const SplitPlan sp = plan_of(n_out, n_in, n_tok, sms);
    const int bn = gemm_bn(n_tok);
    out[0] = sp.S;
    out[1] = sp.m_full;
    out[2] = sp.streamk ? 1 : 0;
    out[3] = (int)(((n_out + GEMM_BM - 1) / GEMM_BM) * ((n_tok + bn - 1) / bn));
}

// Zero the columns of Y that the product's split tiles add into (none when it does not
// split): to be enqueued before the activation conversion (the product kernel overlaps it).
cudaError_t gemm_zero_y(float* Y, int64_t n_out, int64_t n_in, int64_t n_tok, int sms, cudaStream_t s) {
    const SplitPlan sp = plan_of(n_out, n_in, n_tok, sms);
    if (sp.S == 1 && !sp.streamk) return cudaSuccess;
    const int64_t c0 = (int64_t)sp.m_full * GEMM_BM;
    if (c0 == 0) return cudaMemsetAsync(Y, 0, (size_t)n_tok * n_out * sizeof(float), s);
    return cudaMemset2DAsync(Y + c0, (size_t)n_out * sizeof(float), 0, (size_t)(n_out - c0) * sizeof(float),
                             (size_t)n_tok, s);
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
    p.bn = gemm_bn(n_tok);
    p.n_m = (int)((n_out + GEMM_BM - 1) / GEMM_BM);
    p.n_n = (int)((n_tok + p.bn - 1) / p.bn);
    const int64_t tiles = (int64_t)p.n_m * p.n_n;
    if (tiles * 16 > (int64_t(1) << 30) || (int64_t)p.n_super * 16 > (int64_t(1) << 30))
        return cudaErrorInvalidValue;  // 32-bit unit and super-step arithmetic
    const SplitPlan sp = plan_of(n_out, n_in, n_tok, sms);
    p.n_split = sp.S;
    p.m_full = sp.m_full;
    p.u_full = p.m_full * p.n_n;
    p.n_units = (int)((int64_t)p.u_full + ((int64_t)p.n_m - p.m_full) * p.n_n * p.n_split);
    p.accumulate = p.n_split > 1 ? 1 : 0;
    if (sp.streamk) {
        p.sk_tile0 = p.m_full * p.n_n;
        p.streamk_work = (int)((tiles - p.sk_tile0) * p.n_super);
        p.n_units = p.sk_tile0 + p.streamk_work;  // the grid is at most this many CTAs
        p.accumulate = 1;
    }
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

    // weights: one 2-D TMA box (128 rows x BOX bytes) per raw stage when the row pitch
    // allows it (W itself is 16-byte aligned); otherwise per-row copy windows
    int box_bytes, esize, raw_row;
    switch (type) {
    case SYN_Q4_K: box_bytes = GemmFmt<SYN_Q4_K>::BOX; esize = GemmFmt<SYN_Q4_K>::ESIZE; raw_row = GemmFmt<SYN_Q4_K>::RAW_ROW; break;
    case SYN_Q6_K: box_bytes = GemmFmt<SYN_Q6_K>::BOX; esize = GemmFmt<SYN_Q6_K>::ESIZE; raw_row = GemmFmt<SYN_Q6_K>::RAW_ROW; break;
    case SYN_Q8_0: box_bytes = GemmFmt<SYN_Q8_0>::BOX; esize = GemmFmt<SYN_Q8_0>::ESIZE; raw_row = GemmFmt<SYN_Q8_0>::RAW_ROW; break;
    case SYN_Q4_0: box_bytes = GemmFmt<SYN_Q4_0>::BOX; esize = GemmFmt<SYN_Q4_0>::ESIZE; raw_row = GemmFmt<SYN_Q4_0>::RAW_ROW; break;
    case SYN_Q5_0: box_bytes = GemmFmt<SYN_Q5_0>::BOX; esize = GemmFmt<SYN_Q5_0>::ESIZE; raw_row = GemmFmt<SYN_Q5_0>::RAW_ROW; break;
    case SYN_F16: box_bytes = 0; esize = 2; raw_row = 0; break;
    default: return cudaErrorInvalidValue;
    }
    CUtensorMap wmap = map;  // placeholder when unused
    p.raw_tma = 0;
    p.raw_row = raw_row;
    if (type == SYN_F16) {
        // fp16 rows (n_in % 8 == 0): 64-k x 128-row boxes, 128-byte swizzle, as the A tile
        cuuint64_t wdims[2] = {(cuuint64_t)n_in, (cuuint64_t)n_out};
        cuuint64_t wstrides[1] = {(cuuint64_t)n_in * 2};
        cuuint32_t wbox[2] = {(cuuint32_t)GEMM_BK, (cuuint32_t)GEMM_BM};
        cr = encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(W), wdims, wstrides, wbox, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    } else if (p.row_bytes % 16 == 0 && p.row_bytes < (int64_t(1) << 31)) {
        cuuint64_t wdims[2] = {(cuuint64_t)(p.row_bytes / esize), (cuuint64_t)n_out};
        cuuint64_t wstrides[1] = {(cuuint64_t)p.row_bytes};
        cuuint32_t wbox[2] = {(cuuint32_t)(box_bytes / esize), (cuuint32_t)GEMM_BM};
        cr = encode(&wmap, esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                    const_cast<void*>(W), wdims, wstrides, wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
        p.raw_tma = 1;
        p.raw_row = box_bytes;
    }
    // outputs: 2-D TMA box of 32 outputs x 16 tokens when the Y row pitch is a multiple of
    // 16 bytes (Y itself is 16-byte aligned)
    CUtensorMap ymap = map;  // placeholder when unused
    p.y_tma = 0;
    if (n_out % 4 == 0) {
        cuuint64_t ydims[2] = {(cuuint64_t)n_out, (cuuint64_t)n_tok};
        cuuint64_t ystrides[1] = {(cuuint64_t)n_out * 4};
        cuuint32_t ybox[2] = {32, (cuuint32_t)GEMM_OUT_TOK};
        cr = encode(&ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, Y, ydims, ystrides, ybox, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
        p.y_tma = 1;
    }
    switch (type) {
    case SYN_Q4_K: return run_gemm<SYN_Q4_K>(p, map, wmap, ymap, sms, s);
    case SYN_Q6_K: return run_gemm<SYN_Q6_K>(p, map, wmap, ymap, sms, s);
    case SYN_Q8_0: return run_gemm<SYN_Q8_0>(p, map, wmap, ymap, sms, s);
    case SYN_Q4_0: return run_gemm<SYN_Q4_0>(p, map, wmap, ymap, sms, s);
    case SYN_Q5_0: return run_gemm<SYN_Q5_0>(p, map, wmap, ymap, sms, s);
    case SYN_F16: return run_gemm<SYN_F16>(p, map, wmap, ymap, sms, s);
    default: return cudaErrorInvalidValue;
    }
}

#ifdef SYN_DEBUG
SYN_BOUNDS_READER(debug_bounds_gemm)
#endif

}  // namespace syn

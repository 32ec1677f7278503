// common.cuh — block-format constants and sm_103a primitives shared by the kernels.
//
// Block formats: "The GGML ecosystem, and where synapse fits", section 5 (format table).
// In-block byte order is the public GGUF layout:
//   Q8_0 [d f16][q int8 x32]                                          34 B
//   Q4_K [d f16][dmin f16][scales 12 B][q nibbles 128 B]              144 B
//   Q6_K [ql 128 B][qh 64 B][scales int8 x16][d f16]                   210 B
//   Q8_K [d f32][q int8 x256][bsums int16 x16]                         292 B
//   Q4_0 [d f16][qs 16 B: q[l] low nibble, q[l+16] high nibble]       18 B
//   Q5_0 [d f16][qh u32: bit i = fifth bit of q[i]][qs 16 B as Q4_0]   22 B
//   F16  one IEEE half per weight                                     2 B
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#define SYN_Q8_0 1
#define SYN_Q4_K 2
#define SYN_Q6_K 3
#define SYN_Q8_K 4
#define SYN_Q4_0 5
#define SYN_Q5_0 6
#define SYN_F16 7

// Device-side error codes written into the library's per-device error word.
#define SYN_DEVERR_TIMEOUT 1
#define SYN_DEVERR_BOUNDS 2

// Bounded waits: a wait that has not completed after this many clock cycles (about
// two seconds at the maximum SM clock) gives up, records SYN_DEVERR_TIMEOUT and
// returns false so that the kernel can wind down instead of hanging.
#ifndef SYN_WAIT_CYCLES
#define SYN_WAIT_CYCLES (4000000000ll)
#endif
// Bound of a drain: the wait, after a kernel gave up, for copies or tensor-core operations
// it had already issued (they complete on their own; the bound only keeps the wait finite).
#ifndef SYN_DRAIN_CYCLES
#define SYN_DRAIN_CYCLES (4000000000ll)
#endif

namespace syn {

template <int T> struct Fmt;
template <> struct Fmt<SYN_Q8_0> { static constexpr int elems = 32, bytes = 34; };
template <> struct Fmt<SYN_Q4_K> { static constexpr int elems = 256, bytes = 144; };
template <> struct Fmt<SYN_Q6_K> { static constexpr int elems = 256, bytes = 210; };
template <> struct Fmt<SYN_Q8_K> { static constexpr int elems = 256, bytes = 292; };
template <> struct Fmt<SYN_Q4_0> { static constexpr int elems = 32, bytes = 18; };
template <> struct Fmt<SYN_Q5_0> { static constexpr int elems = 32, bytes = 22; };

// 32-weight formats (vec_dot_type Q8_0)
__host__ __device__ inline bool small_block(int t) { return t == SYN_Q8_0 || t == SYN_Q4_0 || t == SYN_Q5_0; }
__host__ __device__ inline int block_elems(int t) { return t == SYN_F16 ? 1 : small_block(t) ? 32 : 256; }
__host__ __device__ inline int block_bytes(int t) {
    return t == SYN_Q8_0 ? 34 : t == SYN_Q4_K ? 144 : t == SYN_Q6_K ? 210 : t == SYN_Q8_K ? 292 : t == SYN_Q4_0 ? 18
         : t == SYN_Q5_0 ? 22 : 2;
}

// ---------------------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ float h2f_bits(uint16_t b) {
    return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Read a 32-bit word from shared memory at any 1-byte offset (two aligned loads and a
// funnel shift; the second load stays inside the allocation when the caller guarantees
// 4 readable bytes past p rounded down).
__device__ __forceinline__ uint32_t lds_u32_any(const uint8_t* p) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    uint32_t sh = static_cast<uint32_t>(a & 3) * 8;
    uint32_t lo = w[0];
    if (sh == 0) return lo;
    return __funnelshift_r(lo, w[1], sh);
}

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

__device__ __forceinline__ void record_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------------------
// Index checks of the SYN_DEBUG build (the stand-in for a memory checker).  SYN_IN_BOUNDS(c)
// guards one access or copy: in the debug build it is c, and a false c records
// SYN_DEVERR_BOUNDS in this translation unit's status word (the library is compiled
// without relocatable device code, so each kernel file has its own word, read by its
// SYN_BOUNDS_READER function) and the caller skips the access.  In other builds it is the
// constant true and compiles away.
// ---------------------------------------------------------------------------------------
#ifdef SYN_DEBUG
static __device__ int g_syn_bounds;
__device__ __forceinline__ bool in_bounds(bool ok) {
    if (!ok) atomicCAS(&g_syn_bounds, 0, SYN_DEVERR_BOUNDS);
    return ok;
}
#define SYN_IN_BOUNDS(cond) (::syn::in_bounds(cond))
// Host function `int name(int clear)`: this file's status word on the current device (and
// reset it when clear != 0); -1 if it cannot be read.
#define SYN_BOUNDS_READER(name)                                                               \
    int name(int clear) {                                                                     \
        int v = 0;                                                                            \
        if (cudaMemcpyFromSymbol(&v, ::syn::g_syn_bounds, sizeof(int)) != cudaSuccess) return -1; \
        const int z = 0;                                                                      \
        if (clear && cudaMemcpyToSymbol(::syn::g_syn_bounds, &z, sizeof(int)) != cudaSuccess) return -1; \
        return v;                                                                             \
    }
#else
#define SYN_IN_BOUNDS(cond) (true)
#endif

// ---------------------------------------------------------------------------------------
// mbarrier / bulk-copy primitives (PTX ISA: mbarrier, cp.async.bulk)
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps in hardware until the phase
// completes or about a microsecond passes, instead of spinning on the issue slots.
#ifndef SYN_WAIT_SLEEP_NS
#define SYN_WAIT_SLEEP_NS 1000
#endif
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    if (SYN_WAIT_SLEEP_NS == 0) return mbar_try_wait(bar, parity);
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"((uint32_t)SYN_WAIT_SLEEP_NS)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// SYN_WAIT_CYCLES, or as soon as *abort is set by another thread of the CTA; on
// giving up it records the timeout, sets *abort and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err,
                                          volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > SYN_WAIT_CYCLES) {
            record_error(err, SYN_DEVERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

// Wait for a phase whose copies (or tensor-core commits) were issued by this CTA, ignoring
// the abort flag: after a kernel gave up, every asynchronous write into its shared memory
// must have landed before the CTA leaves, or it would land in the next CTA's.  Bounded by
// SYN_DRAIN_CYCLES (records SYN_DEVERR_TIMEOUT if it ever runs out).  Returns at once on a
// phase that has completed, as every phase has on the normal path.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, int* err) {
    if (mbar_try_wait(bar, parity)) return;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > SYN_DRAIN_CYCLES) {
            record_error(err, SYN_DEVERR_TIMEOUT);
            return;
        }
    }
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier (bytes).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Signed 4-way byte dot product.  The 4- and 6-bit weight codes (0..63) are below 128,
// so they read the same as signed bytes.
__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// 4-way byte dot product of unsigned bytes a with signed bytes b: for the high nibbles of
// packed codes masked in place (16 x code, up to 240), whose sum is then 16 x the code sum,
// exactly (an arithmetic shift by 4 recovers it).
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

}  // namespace syn

// gemv_f16.cu — decode product for F16 weights: Y[t][o] = sum_i w[o][i] * fp16(x[t][i]).
//
// "The GGML ecosystem, and where synapse fits", section 5: the vec_dot_type of F16 weights
// is F16, i.e. the activations are rounded to fp16 before the product ("Products: weights
// against quantized activations").  Each product of two fp16 values is exact in fp32; the
// sum is accumulated in fp32.  Decode streams every weight once (2 bytes per weight), so
// the kernel is bound by HBM bandwidth: 16-byte loads, four in flight per lane, fp32 FMAs.
#include "common.cuh"
#include "kernels.h"

namespace syn {

constexpr int F16_WARPS = 8;     // warps per CTA
constexpr int F16_UNROLL = 4;    // 16-byte weight loads in flight per lane

// X (n_tok x n_in fp32) -> x16 (n_tok x n_in fp16, round to nearest even); n_in % 8 == 0
__global__ void __launch_bounds__(256) k_x_to_half(const float* __restrict__ X, int64_t n8, __half* __restrict__ xh) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = *reinterpret_cast<const float4*>(X + 8 * i);
        const float4 b = *reinterpret_cast<const float4*>(X + 8 * i + 4);
        const __half2 h0 = __floats2half2_rn(a.x, a.y), h1 = __floats2half2_rn(a.z, a.w);
        const __half2 h2 = __floats2half2_rn(b.x, b.y), h3 = __floats2half2_rn(b.z, b.w);
        uint4 o;
        o.x = *reinterpret_cast<const uint32_t*>(&h0);
        o.y = *reinterpret_cast<const uint32_t*>(&h1);
        o.z = *reinterpret_cast<const uint32_t*>(&h2);
        o.w = *reinterpret_cast<const uint32_t*>(&h3);
        *reinterpret_cast<uint4*>(xh + 8 * i) = o;
    }
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void h8_to_f8(const uint4 v, float f[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// One warp per output row at a time (grid-stride over rows); lane L takes halves 8L..8L+7 of
// every 256-wide slice of the row.
template <int NT>
__global__ void __launch_bounds__(F16_WARPS * 32) k_gemv_f16(const __half* __restrict__ W, int64_t n_out, int n_in,
                                                           const __half* __restrict__ xh, int64_t n_tok,
                                                           float* __restrict__ Y) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * F16_WARPS + (threadIdx.x >> 5);
    const int64_t GW = (int64_t)gridDim.x * F16_WARPS;
    for (int64_t t0 = 0; t0 < n_tok; t0 += NT) {
        for (int64_t o = gw; o < n_out; o += GW) {
            const __half* wr = W + o * n_in;
            float acc[NT];
#pragma unroll
            for (int t = 0; t < NT; t++) acc[t] = 0.f;
            for (int base = 8 * lane; base < n_in; base += 256 * F16_UNROLL) {
                uint4 wv[F16_UNROLL];
#pragma unroll
                for (int u = 0; u < F16_UNROLL; u++)
                    if (base + 256 * u < n_in && SYN_IN_BOUNDS(base + 256 * u + 8 <= n_in))
                        wv[u] = ldg_nc_v4(wr + base + 256 * u);
#pragma unroll
                for (int u = 0; u < F16_UNROLL; u++) {
                    const int k = base + 256 * u;
                    if (k >= n_in) break;
                    float wf[8];
                    h8_to_f8(wv[u], wf);
#pragma unroll
                    for (int t = 0; t < NT; t++) {
                        if (t0 + t >= n_tok) break;
                        float xf[8];
                        h8_to_f8(*reinterpret_cast<const uint4*>(xh + (t0 + t) * n_in + k), xf);
#pragma unroll
                        for (int i = 0; i < 8; i++) acc[t] = fmaf(wf[i], xf[i], acc[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < NT; t++) {
                float v = acc[t];
#pragma unroll
                for (int s = 16; s > 0; s >>= 1) v += __shfl_xor_sync(0xffffffffu, v, s);
                if (lane == 0 && t0 + t < n_tok && SYN_IN_BOUNDS(o < n_out)) Y[(t0 + t) * n_out + o] = v;
            }
        }
    }
}

cudaError_t launch_x_to_half(const float* X, int64_t n, void* xh, int sms, cudaStream_t s) {
    const int64_t n8 = n / 8;
    int64_t g = (n8 + 255) / 256;
    if (g > (int64_t)sms * 8) g = (int64_t)sms * 8;
    if (g < 1) g = 1;
    k_x_to_half<<<(unsigned)g, 256, 0, s>>>(X, n8, static_cast<__half*>(xh));
    return cudaGetLastError();
}

cudaError_t launch_gemv_f16(const void* W, int64_t n_out, int64_t n_in, const float* X, int64_t n_tok, float* Y,
                            void* ws, int sms, cudaStream_t s) {
    cudaError_t e = launch_x_to_half(X, n_tok * n_in, ws, sms, s);
    if (e != cudaSuccess) return e;
    int64_t g = (n_out + F16_WARPS - 1) / F16_WARPS;
    if (g > (int64_t)sms * 8) g = (int64_t)sms * 8;
    const __half* w = static_cast<const __half*>(W);
    const __half* x = static_cast<const __half*>(ws);
    if (n_tok <= 1) k_gemv_f16<1><<<(unsigned)g, F16_WARPS * 32, 0, s>>>(w, n_out, (int)n_in, x, n_tok, Y);
    else if (n_tok <= 2) k_gemv_f16<2><<<(unsigned)g, F16_WARPS * 32, 0, s>>>(w, n_out, (int)n_in, x, n_tok, Y);
    else if (n_tok <= 4) k_gemv_f16<4><<<(unsigned)g, F16_WARPS * 32, 0, s>>>(w, n_out, (int)n_in, x, n_tok, Y);
    else k_gemv_f16<8><<<(unsigned)g, F16_WARPS * 32, 0, s>>>(w, n_out, (int)n_in, x, n_tok, Y);
    return cudaGetLastError();
}

#ifdef SYN_DEBUG
SYN_BOUNDS_READER(debug_bounds_gemv_f16)
#endif

}  // namespace syn

// noalloc.cu — syn_mul_mat_prefill_static: the prefill product with its scratch in a
// fixed device array, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the product: code that
// runs under a custom allocator or a memory budget that forbids the CUDA allocator, code
// inside a pre-planned memory arena, or a runtime that must not synchronise the device
// (cudaMalloc/cudaFree can).  syn_mul_mat's prefill path keeps its fp16 activation
// operand in a workspace the library allocates on first need; this entry point keeps it
// instead in the file-scope array below, loaded with the library on every device that
// uses it and held until the process exits.  It allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "syn.h"

namespace {

// Bytes 0..255: device status word (timeout flag of the product kernels) and padding.
// Bytes 256..: the fp16 activation operand, n_tok * n_in * 2 bytes at most
// SYN_STATIC_SCRATCH_BYTES.
constexpr size_t kHeader = 256;
static __device__ __align__(256) unsigned char g_scratch[kHeader + SYN_STATIC_SCRATCH_BYTES];

struct StaticDevice {
    bool ready = false;
    int sms = 0;
    unsigned char* scratch = nullptr;  // device address of g_scratch on this device
};

std::mutex g_mu;
StaticDevice g_devices[64];

// Once per device, with that device current: the device address of the array (the host
// symbol g_scratch is only a stand-in and must never be handed to a kernel), the SM count,
// and a cleared status word.  Must run before any stream capture that contains this call.
int setup(int dev, StaticDevice** out) {
    if (dev < 0 || dev >= 64) return SYN_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    StaticDevice& d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SYN_ERR_CUDA;
        if (major != 10 || minor != 3) return SYN_ERR_DEVICE;
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) return SYN_ERR_CUDA;
        if (cudaMemset(ptr, 0, kHeader) != cudaSuccess) return SYN_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return SYN_ERR_CUDA;
        d.scratch = static_cast<unsigned char*>(ptr);
        d.sms = sms;
        d.ready = true;
    }
    *out = &d;
    return SYN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

namespace syn {

// Read (and optionally reset) the status word at the head of the fixed array; a device
// that has not run syn_mul_mat_prefill_static has none and reads as 0.
int static_status(int dev, int clear, int* word) {
    *word = 0;
    if (dev < 0 || dev >= 64) return SYN_OK;
    std::lock_guard<std::mutex> lk(g_mu);
    const StaticDevice& d = g_devices[dev];
    if (!d.ready) return SYN_OK;
    if (cudaMemcpy(word, d.scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SYN_ERR_CUDA;
    if (clear && cudaMemset(d.scratch, 0, sizeof(int)) != cudaSuccess) return SYN_ERR_CUDA;
    return SYN_OK;
}

}  // namespace syn

extern "C" int syn_mul_mat_prefill_static(int type, const void* W, int64_t n_out, int64_t n_in, const float* X,
                                          int64_t n_tok, float* Y, syn_stream_t stream) {
    if (type < SYN_TYPE_Q8_0 || type > SYN_TYPE_F16 || type == SYN_TYPE_Q8_K) return SYN_ERR_TYPE;
    const int64_t be = syn::block_elems(type);
    // F16 rows are read 16 bytes (8 values) at a time, as in syn_mul_mat
    const int64_t row_multiple = type == SYN_TYPE_F16 ? 8 : be;
    if (n_out <= 0 || n_in <= 0 || n_tok < 0 || n_in % row_multiple || n_out > (int64_t(1) << 31) ||
        n_out * n_in > (int64_t(1) << 40) || n_tok * n_out > (int64_t(1) << 40))
        return SYN_ERR_SHAPE;
    if (n_tok > (int64_t)(SYN_STATIC_SCRATCH_BYTES / 2) / n_in) return SYN_ERR_TOO_LARGE;
    if (n_tok == 0) return SYN_OK;
    if (!W || !X || !Y) return SYN_ERR_NULL;
    if (!aligned16(W) || !aligned16(X) || !aligned16(Y)) return SYN_ERR_ALIGN;
    int dev;
    if (cudaGetDevice(&dev) != cudaSuccess) return SYN_ERR_CUDA;
    StaticDevice* d;
    int rc = setup(dev, &d);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int lim = syn::sm_limit();
    const int sms = lim > 0 && lim < d->sms ? lim : d->sms;
    int* err = reinterpret_cast<int*>(d->scratch);
    void* xh = d->scratch + kHeader;
    const int xt = (type == SYN_TYPE_Q4_K || type == SYN_TYPE_Q6_K) ? SYN_TYPE_Q8_K
                 : type == SYN_TYPE_F16 ? SYN_TYPE_F16 : SYN_TYPE_Q8_0;
    if (syn::gemm_zero_y(Y, n_out, n_in, n_tok, sms, s) != cudaSuccess) return SYN_ERR_CUDA;
    if (syn::launch_act_half(xt, X, n_tok * (n_in / be), xh, sms, s) != cudaSuccess) return SYN_ERR_CUDA;
    syn::note_launches(1);
    if (syn::launch_gemm(type, W, n_out, n_in, xh, n_tok, Y, err, sms, s) != cudaSuccess) return SYN_ERR_CUDA;
    syn::note_launches(1);
    return SYN_OK;
}

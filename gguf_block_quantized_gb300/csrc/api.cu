// api.cu — the C ABI of libsyn (declared in include/syn.h): argument checks, dispatch to
// the kernels, the per-(device, stream) prefill workspace and the device status words.
//
// Conventions follow "The GGML ecosystem, and where synapse fits": unsupported input is
// rejected, never approximated (section 1, and the synapse table in section 7); untrusted
// input is validated without exceptions; the matrix orientation is ggml_mul_mat's
// (yakaai ggml documentation, examples/simple).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <map>
#include <vector>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "kernels.h"
#include "syn.h"

namespace {

using syn::launch_act_half;

std::atomic<long long> g_launches{0};
// Decode/prefill threshold: -1 = per format (decode_max_tok), else the same n for every
// format (syn_set_gemv_max_tok, or SYN_GEMV_MAX_TOK in the environment at load time)
std::atomic<int> g_gemv_max_tok{[] {
    const char* e = std::getenv("SYN_GEMV_MAX_TOK");
    if (e && *e) {
        char* end = nullptr;
        long v = std::strtol(e, &end, 10);
        if (end && *end == 0 && v >= 0 && v < (1 << 30)) return (int)v;
    }
    return -1;
}()};

// Largest n_tok that runs on the decode kernels.  Per format, the measured crossover with
// the tensor-core prefill on GB300 (decode re-reads the weights per group of 8 tokens and
// its per-token work is larger for the 32-weight formats and F16): K-quants 8, Q8_0 / Q4_0
// / Q5_0 4, F16 2.
int decode_max_tok(int type) {
    const int v = g_gemv_max_tok.load();
    if (v >= 0) return v;
    if (type == SYN_TYPE_Q4_K || type == SYN_TYPE_Q6_K) return 8;
    if (type == SYN_TYPE_F16) return 2;
    return 4;
}

// Prefill calls of at least this many tokens expand Q6_K weights (Q4_K: twice as many) to
// fp16 once per product (launch_deq_half) and run the fp16 tensor-core product on them: the
// fused product expands every weight tile again for each 256-token tile, and from about this
// size that costs more than one pass over the weights (measured on GB300, 2048 tokens: Q6_K
// FFN down 4096x14336 275.0 us fused, 252.9 us expanded; at 512 tokens the fused product
// wins).  syn_set_prefill_expand_tok, or SYN_PREFILL_EXPAND_TOK at load time.
#ifndef SYN_PREFILL_EXPAND_TOK_DEFAULT
#define SYN_PREFILL_EXPAND_TOK_DEFAULT 1536
#endif
constexpr int kPrefillExpandTok = SYN_PREFILL_EXPAND_TOK_DEFAULT;
std::atomic<int> g_expand_tok{[] {
    const char* e = std::getenv("SYN_PREFILL_EXPAND_TOK");
    if (e && *e) {
        char* end = nullptr;
        long v = std::strtol(e, &end, 10);
        if (end && *end == 0 && v >= 0 && v < (1 << 30)) return (int)v;
    }
    return kPrefillExpandTok;
}()};

std::atomic<int> g_det{0};       // deterministic mode (syn_set_deterministic)
std::atomic<int> g_sm_limit{0};  // 0: every SM

struct DeviceState {
    bool init = false;
    int sms = 0;
    int* words = nullptr;  // [0] timeout/error word, [1] quantize range flag
};

struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};

std::mutex g_mu;
std::map<int, DeviceState> g_dev;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

int current_device(int* dev) {
    return cudaGetDevice(dev) == cudaSuccess ? SYN_OK : SYN_ERR_CUDA;
}

// Per-device state: SM count, capability check, the two status words.
int device_state(DeviceState** out) {
    int dev;
    if (current_device(&dev) != SYN_OK) return SYN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SYN_ERR_CUDA;
        if (major != 10 || minor != 3) return SYN_ERR_DEVICE;  // built for sm_103a only
        int* w = nullptr;
        if (cudaMalloc(&w, 2 * sizeof(int)) != cudaSuccess) return SYN_ERR_NOMEM;
        if (cudaMemset(w, 0, 2 * sizeof(int)) != cudaSuccess) return SYN_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return SYN_ERR_CUDA;
        st.sms = sms;
        st.words = w;
        st.init = true;
    }
    *out = &st;
    return SYN_OK;
}

// SMs the launches of this call may use.
int sms_of(const DeviceState* st) {
    const int lim = g_sm_limit.load();
    return lim > 0 && lim < st->sms ? lim : st->sms;
}

}  // namespace

namespace syn {
int sm_limit() { return g_sm_limit.load(); }
}  // namespace syn

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool known_type(int t) { return t >= SYN_TYPE_Q8_0 && t <= SYN_TYPE_F16; }
// weight formats of mul_mat (Q8_K is an activation format only)
bool is_weight(int t) { return known_type(t) && t != SYN_TYPE_Q8_K; }
// the vec_dot_type the activations are converted to: Q8_0 for the 32-weight formats,
// Q8_K for the K-quants, F16 for F16 ("Products: weights against quantized activations")
int vec_dot(int t) {
    return (t == SYN_TYPE_Q4_K || t == SYN_TYPE_Q6_K) ? SYN_TYPE_Q8_K : t == SYN_TYPE_F16 ? SYN_TYPE_F16 : SYN_TYPE_Q8_0;
}


int64_t elems(int t) { return syn::block_elems(t); }
int64_t bytes_of(int t) { return syn::block_bytes(t); }
// F16 rows are read 8 values (16 bytes) at a time
int64_t row_multiple(int t) { return t == SYN_TYPE_F16 ? 8 : elems(t); }

int check_cuda(cudaError_t e) { return e == cudaSuccess ? SYN_OK : SYN_ERR_CUDA; }

// Largest shapes a single call may take (int32 index arithmetic inside the kernels stays
// far from overflow within these limits).
constexpr int64_t kMaxElems = int64_t(1) << 40;

// Prefill workspace bytes: the fp16 activation operand.
size_t prefill_ws_bytes(int64_t n_in, int64_t n_tok) { return (size_t)(n_in * n_tok * 2 + 256); }

int workspace_for(cudaStream_t s, size_t need, void** out) {
    int dev;
    if (current_device(&dev) != SYN_OK) return SYN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace& w = g_ws[{dev, s}];
    if (w.bytes < need) {
        if (w.ptr) {
            if (cudaDeviceSynchronize() != cudaSuccess) return SYN_ERR_CUDA;
            cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
        }
        if (cudaMalloc(&w.ptr, need) != cudaSuccess) {
            (void)cudaGetLastError();  // not sticky: keep it out of the next launch check
            w.ptr = nullptr;
            return SYN_ERR_NOMEM;
        }
        w.bytes = need;
    }
    *out = w.ptr;
    return SYN_OK;
}

}  // namespace

namespace syn {
void note_launches(int n) { g_launches += n; }
}  // namespace syn

extern "C" {

int64_t syn_block_elems(int type) { return known_type(type) ? elems(type) : -1; }

int64_t syn_block_bytes(int type) { return known_type(type) ? bytes_of(type) : -1; }

int64_t syn_row_bytes(int type, int64_t n) {
    if (!known_type(type) || n <= 0 || n % elems(type)) return -1;
    return n / elems(type) * bytes_of(type);
}

const char* syn_strerror(int status) {
    switch (status) {
    case SYN_OK: return "ok";
    case SYN_ERR_TYPE: return "unknown or unsupported block format";
    case SYN_ERR_SHAPE: return "bad shape (size <= 0 or not a multiple of the block size)";
    case SYN_ERR_NULL: return "null pointer";
    case SYN_ERR_ALIGN: return "pointer not 16-byte aligned";
    case SYN_ERR_RANGE: return "non-finite input or scale out of fp16 range";
    case SYN_ERR_CUDA: return "CUDA error";
    case SYN_ERR_TIMEOUT: return "a device-side wait timed out";
    case SYN_ERR_NOMEM: return "out of device memory";
    case SYN_ERR_DEVICE: return "device is not sm_103 (GB300)";
    case SYN_ERR_TOO_LARGE: return "problem larger than the fixed scratch array";
    case SYN_ERR_FORMAT: return "malformed GGUF file";
    case SYN_ERR_IO: return "file could not be opened, mapped or written";
    case SYN_ERR_NOTFOUND: return "no such GGUF key or tensor";
    case SYN_ERR_BOUNDS: return "a kernel index check failed (SYN_DEBUG build)";
    default: return "unknown status";
    }
}

int64_t syn_launch_count(void) { return g_launches.load(); }

int syn_set_gemv_max_tok(int n) { return g_gemv_max_tok.exchange(n < 0 ? -1 : n); }

int syn_set_deterministic(int on) { return g_det.exchange(on ? 1 : 0); }

int syn_debug_prefill_plan(int64_t n_out, int64_t n_in, int64_t n_tok, int sms, int* out) {
    if (n_out <= 0 || n_in <= 0 || n_tok <= 0 || sms <= 0 || n_out > (int64_t(1) << 31) || n_in > kMaxElems ||
        n_tok > kMaxElems)
        return SYN_ERR_SHAPE;
    if (!out) return SYN_ERR_NULL;
    syn::gemm_plan(n_out, n_in, n_tok, sms, out);
    return SYN_OK;
}

int syn_set_prefill_expand_tok(int n) { return g_expand_tok.exchange(n < 0 ? kPrefillExpandTok : n); }

int syn_set_sm_limit(int n) {
    if (n < 0) return -1;
    return g_sm_limit.exchange(n);
}

int syn_quantize(int type, const float* src, void* dst, int64_t n_rows, int64_t n_per_row, syn_stream_t stream) {
    if (!known_type(type)) return SYN_ERR_TYPE;
    if (n_rows < 0 || n_per_row <= 0 || n_per_row % elems(type) || n_rows * n_per_row > kMaxElems)
        return SYN_ERR_SHAPE;
    if (n_rows == 0) return SYN_OK;
    if (!src || !dst) return SYN_ERR_NULL;
    if (!aligned16(src) || !aligned16(dst)) return SYN_ERR_ALIGN;
    DeviceState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int* range = st->words + 1;
    if (cudaMemsetAsync(range, 0, sizeof(int), s) != cudaSuccess) return SYN_ERR_CUDA;
    const int64_t nblocks = n_rows * (n_per_row / elems(type));
    if (syn::launch_quantize(type, src, dst, nblocks, range, sms_of(st), s) != cudaSuccess) return SYN_ERR_CUDA;
    g_launches++;
    int flag = 0;
    if (cudaMemcpyAsync(&flag, range, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SYN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SYN_ERR_CUDA;
    return flag ? SYN_ERR_RANGE : SYN_OK;
}

int syn_dequantize(int type, const void* src, float* dst, int64_t n_rows, int64_t n_per_row, syn_stream_t stream) {
    if (!known_type(type)) return SYN_ERR_TYPE;
    if (n_rows < 0 || n_per_row <= 0 || n_per_row % elems(type) || n_rows * n_per_row > kMaxElems)
        return SYN_ERR_SHAPE;
    if (n_rows == 0) return SYN_OK;
    if (!src || !dst) return SYN_ERR_NULL;
    if (!aligned16(src) || !aligned16(dst)) return SYN_ERR_ALIGN;
    DeviceState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    const int64_t nblocks = n_rows * (n_per_row / elems(type));
    if (syn::launch_dequantize(type, src, dst, nblocks, sms_of(st), reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SYN_ERR_CUDA;
    g_launches++;
    return SYN_OK;
}

int syn_dequantize_f16(int type, const void* src, void* dst, int64_t n_rows, int64_t n_per_row, syn_stream_t stream) {
    if (type != SYN_TYPE_Q4_K && type != SYN_TYPE_Q6_K) return SYN_ERR_TYPE;
    if (n_rows < 0 || n_per_row <= 0 || n_per_row % elems(type) || n_rows * n_per_row > kMaxElems)
        return SYN_ERR_SHAPE;
    if (n_rows == 0) return SYN_OK;
    if (!src || !dst) return SYN_ERR_NULL;
    if (!aligned16(src) || !aligned16(dst)) return SYN_ERR_ALIGN;
    DeviceState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    const int64_t nblocks = n_rows * (n_per_row / elems(type));
    if (syn::launch_deq_half(type, src, dst, nblocks, sms_of(st), reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SYN_ERR_CUDA;
    g_launches++;
    return SYN_OK;
}

int syn_quantize_activations(int wtype, const float* X, int64_t n_tok, int64_t n_in, int8_t* qs, float* d,
                             int16_t* bsums, syn_stream_t stream) {
    if (!is_weight(wtype) || wtype == SYN_TYPE_F16) return SYN_ERR_TYPE;  // F16: syn_quantize(F16, X)
    const int xt = vec_dot(wtype);
    if (n_tok < 0 || n_in <= 0 || n_in % elems(xt) || n_tok * n_in > kMaxElems) return SYN_ERR_SHAPE;
    if (n_tok == 0) return SYN_OK;
    if (!X || !qs || !d || (xt == SYN_TYPE_Q8_K && !bsums)) return SYN_ERR_NULL;
    if (!aligned16(X) || !aligned16(qs) || !aligned16(d) || (bsums && !aligned16(bsums))) return SYN_ERR_ALIGN;
    DeviceState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    const int64_t nblocks = n_tok * (n_in / elems(xt));
    if (syn::launch_quantize_act(xt, X, nblocks, qs, d, xt == SYN_TYPE_Q8_K ? bsums : nullptr, sms_of(st),
                                 reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SYN_ERR_CUDA;
    g_launches++;
    return SYN_OK;
}

int syn_reserve(int64_t max_n_in, int64_t max_n_tok, syn_stream_t stream) {
    if (max_n_in <= 0 || max_n_tok < 0 || max_n_in * max_n_tok > kMaxElems) return SYN_ERR_SHAPE;
    DeviceState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    void* p;
    return workspace_for(reinterpret_cast<cudaStream_t>(stream), prefill_ws_bytes(max_n_in, max_n_tok), &p);
}

int syn_release(void) {
    int dev;
    if (current_device(&dev) != SYN_OK) return SYN_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return SYN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto it = g_ws.begin(); it != g_ws.end();) {
        if (it->first.first == dev) {
            cudaFree(it->second.ptr);
            it = g_ws.erase(it);
        } else {
            ++it;
        }
    }
    return SYN_OK;
}

}  // extern "C"

namespace {

// The prefill path of products that share one activation input (the same X, n_in and
// vec_dot_type: q/k/v, or gate/up, of a layer): the Y columns of split tiles zeroed,
// X converted once into the workspace, then one tensor-core launch per product.  At
// g_expand_tok tokens or more, each K-quant product's weights are first expanded to fp16
// (into the workspace after x~, reused product by product) and the product runs on them.
// Order: the first expansion, the conversion, the first product, then expansion and product
// for each further one.  A product kernel starts its weight loads before it waits for the
// launch it follows, so it must follow the conversion (which writes only x~) or a finished
// expansion (launch_deq_half does not release its dependents early).
int prefill_group(const syn_mat_desc* const* g, int m, int64_t n_tok, const DeviceState* st, cudaStream_t s) {
    const int64_t n_in = g[0]->n_in;
    const int xt = vec_dot(g[0]->type);
    // Q6_K from the threshold; Q4_K, whose fused expansion is cheaper, from twice it, and rows
    // longer than 8192 never.  Measured at 2048 tokens (µs, fused / expanded): Q6_K FFN down
    // 275.0 / 252.9, Q6_K lm_head 2197.5 / 1814.0; Q4_K FFN up 190.2 / 192.8, q 73.6 / 77.0,
    // FFN down 208.3 / 207.6 at 2048 but 210.7 / 235.0 in another run (the fp16-weight product
    // of that shape is slow to fill its last wave).
    bool room = true;  // false: the workspace could not take the expanded weights
    auto expand = [&](const syn_mat_desc* d) {
        const int64_t t = g_expand_tok.load();
        return room && ((d->type == SYN_TYPE_Q6_K && n_tok >= t) ||
                        (d->type == SYN_TYPE_Q4_K && n_in <= 8192 && n_tok >= 2 * t));
    };
    const size_t x_bytes = (prefill_ws_bytes(n_in, n_tok) + 255) & ~size_t(255);
    size_t w_bytes = 0;
    for (int i = 0; i < m; i++)
        if (expand(g[i])) w_bytes = std::max(w_bytes, (size_t)(g[i]->n_out * n_in) * 2);
    void* ws;
    int rc = workspace_for(s, x_bytes + w_bytes, &ws);
    if (rc == SYN_ERR_NOMEM && w_bytes > 0) {
        // no room for the expanded weights: the fused product needs only x~
        w_bytes = 0;
        room = false;
        rc = workspace_for(s, x_bytes, &ws);
    }
    if (rc) return rc;
    void* wh = static_cast<uint8_t*>(ws) + x_bytes;
    for (int i = 0; i < m; i++)
        if (syn::gemm_zero_y(g[i]->Y, g[i]->n_out, n_in, n_tok, sms_of(st), s) != cudaSuccess) return SYN_ERR_CUDA;
    for (int i = 0; i < m; i++) {
        int type = g[i]->type;
        const void* W = g[i]->W;
        if (expand(g[i])) {
            if (syn::launch_deq_half(type, W, wh, g[i]->n_out * (n_in / elems(type)), sms_of(st), s) != cudaSuccess)
                return SYN_ERR_CUDA;
            g_launches++;
            type = SYN_TYPE_F16;
            W = wh;
        }
        if (i == 0) {
            if (launch_act_half(xt, g[0]->X, n_tok * (n_in / elems(xt)), ws, sms_of(st), s) != cudaSuccess)
                return SYN_ERR_CUDA;
            g_launches++;
        }
        if (syn::launch_gemm(type, W, g[i]->n_out, n_in, ws, n_tok, g[i]->Y, st->words, sms_of(st), s) != cudaSuccess)
            return SYN_ERR_CUDA;
        g_launches++;
    }
    return SYN_OK;
}

}  // namespace

extern "C" {

int syn_mul_mat(int type, const void* W, int64_t n_out, int64_t n_in, const float* X, int64_t n_tok, float* Y,
                syn_stream_t stream) {
    if (!is_weight(type)) return SYN_ERR_TYPE;
    if (n_out <= 0 || n_in <= 0 || n_tok < 0 || n_in % row_multiple(type) || n_out * n_in > kMaxElems ||
        n_tok * n_in > kMaxElems || n_tok * n_out > kMaxElems || n_out > (int64_t(1) << 31))
        return SYN_ERR_SHAPE;
    if (n_tok == 0) return SYN_OK;
    if (!W || !X || !Y) return SYN_ERR_NULL;
    if (!aligned16(W) || !aligned16(X) || !aligned16(Y)) return SYN_ERR_ALIGN;
    DeviceState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool det = g_det.load() != 0;
    if (type == SYN_TYPE_F16 && (det || n_tok <= decode_max_tok(type))) {
        void* ws;
        rc = workspace_for(s, (size_t)(n_tok * n_in * 2 + 256), &ws);
        if (rc) return rc;
        rc = check_cuda(syn::launch_gemv_f16(W, n_out, n_in, X, n_tok, Y, ws, sms_of(st), s));
        if (rc == SYN_OK) g_launches += 2;
        return rc;
    }
    const bool fits = syn::gemv_act_bytes(type, n_in) <= syn::gemv_act_limit();
    if (det && !fits) return SYN_ERR_SHAPE;
    if (det || (n_tok <= decode_max_tok(type) && fits)) {
        const syn::GemvDesc d{type, W, n_out, n_in, X, Y};
        void* ws;
        rc = workspace_for(s, (size_t)syn::gemv_workspace_bytes(1, &d, n_tok), &ws);
        if (rc) return rc;
        rc = check_cuda(syn::launch_gemv_batch(1, &d, n_tok, ws, st->words, sms_of(st), det, s));
        if (rc == SYN_OK) g_launches += 2;
        return rc;
    }
    const syn_mat_desc d{type, W, n_out, n_in, X, Y};
    const syn_mat_desc* g = &d;
    return prefill_group(&g, 1, n_tok, st, s);
}

}  // extern "C"

namespace {

// Argument checks of syn_mul_mat_batch (SYN_OK also for the no-op n == 0 or n_tok == 0).
int check_batch(int n, const syn_mat_desc* descs, int64_t n_tok) {
    if (n < 0 || n_tok < 0) return SYN_ERR_SHAPE;
    if (n == 0 || n_tok == 0) return SYN_OK;
    if (!descs) return SYN_ERR_NULL;
    for (int i = 0; i < n; i++) {
        const syn_mat_desc& d = descs[i];
        if (!is_weight(d.type)) return SYN_ERR_TYPE;
        if (d.n_out <= 0 || d.n_in <= 0 || d.n_in % row_multiple(d.type) || d.n_out * d.n_in > kMaxElems ||
            n_tok * d.n_in > kMaxElems || n_tok * d.n_out > kMaxElems || d.n_out > (int64_t(1) << 31))
            return SYN_ERR_SHAPE;
        if (!d.W || !d.X || !d.Y) return SYN_ERR_NULL;
        if (!aligned16(d.W) || !aligned16(d.X) || !aligned16(d.Y)) return SYN_ERR_ALIGN;
    }
    // deterministic mode runs every quantized product on the decode kernel: a row too wide
    // for its shared memory is rejected here, before any product of the call is enqueued
    if (g_det.load())
        for (int i = 0; i < n; i++)
            if (descs[i].type != SYN_TYPE_F16 &&
                syn::gemv_act_bytes(descs[i].type, descs[i].n_in) > syn::gemv_act_limit())
                return SYN_ERR_SHAPE;
    return SYN_OK;
}

}  // namespace

extern "C" {

int syn_mul_mat_batch(int n, const syn_mat_desc* descs, int64_t n_tok, syn_stream_t stream) {
    const int ck = check_batch(n, descs, n_tok);
    if (ck || n == 0 || n_tok == 0) return ck;
    DeviceState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool det = g_det.load() != 0;
    // pack the products into launches within the decode kernel's activation and job limits
    syn::GemvDesc group[syn::GEMV_MAX_JOBS];
    int ng = 0;
    int64_t act = 0;
    auto flush = [&]() -> int {
        if (ng == 0) return SYN_OK;
        void* ws;
        int r = workspace_for(s, (size_t)syn::gemv_workspace_bytes(ng, group, n_tok), &ws);
        if (r) return r;
        r = check_cuda(syn::launch_gemv_batch(ng, group, n_tok, ws, st->words, sms_of(st), det, s));
        if (r == SYN_OK) g_launches += 2;
        ng = 0;
        act = 0;
        return r;
    };
    std::vector<const syn_mat_desc*> pre;  // products on the tensor-core prefill path
    for (int i = 0; i < n; i++) {
        const syn_mat_desc& d = descs[i];
        const int64_t a = d.type == SYN_TYPE_F16 ? 0 : syn::gemv_act_bytes(d.type, d.n_in);
        if (!det && (n_tok > decode_max_tok(d.type) || a > syn::gemv_act_limit())) {
            pre.push_back(&d);
            continue;
        }
        // F16 decode, or a row too wide for the decode kernel in deterministic mode: its own call
        if (d.type == SYN_TYPE_F16 || a > syn::gemv_act_limit()) {
            rc = syn_mul_mat(d.type, d.W, d.n_out, d.n_in, d.X, n_tok, d.Y, stream);
            if (rc) return rc;
            continue;
        }
        if (ng == syn::GEMV_MAX_JOBS || act + a > syn::gemv_act_limit()) {
            rc = flush();
            if (rc) return rc;
        }
        group[ng++] = syn::GemvDesc{d.type, d.W, d.n_out, d.n_in, d.X, d.Y};
        act += a;
    }
    rc = flush();
    if (rc) return rc;
    // prefill products grouped by activation input, each group converting its input once
    std::vector<char> done(pre.size(), 0);
    std::vector<const syn_mat_desc*> g;
    for (size_t i = 0; i < pre.size(); i++) {
        if (done[i]) continue;
        g.clear();
        for (size_t j = i; j < pre.size(); j++) {
            if (done[j] || pre[j]->X != pre[i]->X || pre[j]->n_in != pre[i]->n_in ||
                vec_dot(pre[j]->type) != vec_dot(pre[i]->type))
                continue;
            g.push_back(pre[j]);
            done[j] = 1;
        }
        rc = prefill_group(g.data(), (int)g.size(), n_tok, st, s);
        if (rc) return rc;
    }
    return SYN_OK;
}

int syn_mul_mat_batch_staged(int n, const syn_mat_desc* descs, int64_t n_tok, const void* x_host, void* x_dev,
                             size_t x_bytes, const void* y_dev, void* y_host, size_t y_bytes, syn_stream_t stream) {
    const int ck = check_batch(n, descs, n_tok);
    if (ck) return ck;
    if ((x_bytes && (!x_host || !x_dev)) || (y_bytes && (!y_dev || !y_host))) return SYN_ERR_NULL;
    if (n > 0 && n_tok > 0) {  // the device checks of syn_mul_mat_batch, before the copy
        DeviceState* st;
        const int rc = device_state(&st);
        if (rc) return rc;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (x_bytes && cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return SYN_ERR_CUDA;
    const int rc = syn_mul_mat_batch(n, descs, n_tok, stream);
    if (rc) return rc;
    if (y_bytes && cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SYN_ERR_CUDA;
    return SYN_OK;
}

int syn_block_sums(int type, const void* W, int64_t n_out, int64_t n_in, const void* Xq, int64_t n_tok, int32_t* S,
                   syn_stream_t stream) {
    if (!is_weight(type) || type == SYN_TYPE_F16) return SYN_ERR_TYPE;  // F16 products are not integer
    if (n_out <= 0 || n_in <= 0 || n_tok < 0 || n_in % elems(type) || n_out * n_in > kMaxElems ||
        n_tok * n_out * (n_in / elems(type)) > kMaxElems)
        return SYN_ERR_SHAPE;
    if (n_tok == 0) return SYN_OK;
    if (!W || !Xq || !S) return SYN_ERR_NULL;
    DeviceState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    if (syn::launch_block_sums(type, W, n_out, n_in / elems(type), Xq, n_tok, S,
                               reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SYN_ERR_CUDA;
    g_launches++;
    return SYN_OK;
}

int syn_device_status(int clear) {
    // Two words can hold a timeout: the per-device word of the allocating entry points and
    // the one at the head of syn_mul_mat_prefill_static's fixed array.  Neither is created
    // here, so a caller of the static entry point alone still allocates nothing.
    int dev;
    if (current_device(&dev) != SYN_OK) return SYN_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return SYN_ERR_CUDA;
    int* words = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_dev.find(dev);
        if (it != g_dev.end() && it->second.init) words = it->second.words;
    }
    int w = 0, ws = 0;
    if (words) {
        if (cudaMemcpy(&w, words, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SYN_ERR_CUDA;
        if (clear && cudaMemset(words, 0, sizeof(int)) != cudaSuccess) return SYN_ERR_CUDA;
    }
    const int rc = syn::static_status(dev, clear, &ws);
    if (rc) return rc;
#ifdef SYN_DEBUG
    // the index-check words of the kernel files (a failed check outranks a timeout it caused)
    int wb = 0;
    for (int v : {syn::debug_bounds_quant(clear), syn::debug_bounds_gemv(clear), syn::debug_bounds_gemv_f16(clear),
                  syn::debug_bounds_gemm(clear)}) {
        if (v < 0) return SYN_ERR_CUDA;
        wb |= v;
    }
    if (wb) return SYN_ERR_BOUNDS;
#endif
    return (w || ws) ? SYN_ERR_TIMEOUT : SYN_OK;
}

int syn_debug_bounds_selftest(syn_stream_t stream) {
#ifdef SYN_DEBUG
    return syn::launch_bounds_selftest(reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? SYN_OK : SYN_ERR_CUDA;
#else
    (void)stream;
    return 1;
#endif
}

}  // extern "C"

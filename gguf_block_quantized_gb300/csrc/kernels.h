// kernels.h — host-side launchers of the libsyn kernels (internal to the library).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace syn {

cudaError_t launch_quantize(int type, const float* src, void* dst, int64_t n_blocks, int* range_err,
                            int sms, cudaStream_t s);
cudaError_t launch_dequantize(int type, const void* src, float* dst, int64_t n_blocks, int sms,
                              cudaStream_t s);
cudaError_t launch_quantize_act(int xtype, const float* X, int64_t n_blocks, int8_t* qs, float* d,
                                int16_t* bsums, int sms, cudaStream_t s);
cudaError_t launch_act_half(int xtype, const float* X, int64_t n_blocks, void* xh, int sms,
                            cudaStream_t s);
// Q4_K / Q6_K weights -> fp16 values (n_blocks blocks, 256 halves each, row-major like W),
// each the fp32 dequantization rounded once to fp16.
cudaError_t launch_deq_half(int type, const void* src, void* dst, int64_t n_blocks, int sms, cudaStream_t s);
cudaError_t launch_block_sums(int type, const void* W, int64_t n_out, int64_t nb, const void* Xq,
                              int64_t n_tok, int32_t* S, cudaStream_t s);

// Decode products of up to GEMV_MAX_JOBS independent matrices in one launch.
constexpr int GEMV_MAX_JOBS = 16;
struct GemvDesc {
    int type;
    const void* W;
    int64_t n_out, n_in;
    const float* X;
    float* Y;
};
// Decode products: Y = W * Xq for few tokens.  Two launches: the activation conversion into
// the workspace ws (gemv_workspace_bytes), then the decode kernel as its programmatic
// dependent (it streams weights before waiting for the conversion).  no_split: every output
// row is computed by one warp (the deterministic mode), else long rows may be split.
cudaError_t launch_gemv_batch(int n, const GemvDesc* d, int64_t n_tok, void* ws, int* err, int sms, bool no_split,
                              cudaStream_t s);
int64_t gemv_workspace_bytes(int n, const GemvDesc* d, int64_t n_tok);

// Shared memory one token of a matrix's converted activations takes in the decode kernel;
// a launch holds at most gemv_act_limit() bytes of them (all matrices, one token).
int64_t gemv_act_bytes(int type, int64_t n_in);
int64_t gemv_act_limit();

// The SM limit set by syn_set_sm_limit (0: none).
int sm_limit();

// Prefill product on the tensor cores.  xh: n_tok x n_in fp16 activations, written by
// launch_act_half immediately before on the same stream (the product kernel is its
// programmatic dependent).  Y is overwritten, except where the product splits along K: those
// columns are added into, so the caller enqueues gemm_zero_y() before launch_act_half.
cudaError_t launch_gemm(int type, const void* W, int64_t n_out, int64_t n_in, const void* xh,
                        int64_t n_tok, float* Y, int* err, int sms, cudaStream_t s);
cudaError_t gemm_zero_y(float* Y, int64_t n_out, int64_t n_in, int64_t n_tok, int sms, cudaStream_t s);
// The prefill schedule of a product (host only): {S, m_full, stream-K, tiles}.
void gemm_plan(int64_t n_out, int64_t n_in, int64_t n_tok, int sms, int out[4]);

// F16 weights (n_in % 8 == 0): X -> fp16 (round to nearest even) into xh, and the decode
// product reading W and the fp16 activations from ws (n_tok * n_in halves).
cudaError_t launch_x_to_half(const float* X, int64_t n, void* xh, int sms, cudaStream_t s);
cudaError_t launch_gemv_f16(const void* W, int64_t n_out, int64_t n_in, const float* X, int64_t n_tok, float* Y,
                            void* ws, int sms, cudaStream_t s);

// Adds n to the count syn_launch_count reports.
void note_launches(int n);

// The status word of syn_mul_mat_prefill_static's fixed array on device dev: *word gets it
// (0 when that entry point has not run on dev); clear != 0 resets it.  Allocates nothing;
// the caller synchronizes the device first.
int static_status(int dev, int clear, int* word);

#ifdef SYN_DEBUG
// SYN_DEBUG build: the index-check status word of each kernel file on the current device
// (SYN_DEVERR_BOUNDS when a check failed; -1 if unreadable), reset when clear != 0, and a
// launch whose one check is given an out-of-range index on purpose (the access it guards,
// into a shared array twice the checked size, is skipped).
int debug_bounds_quant(int clear);
int debug_bounds_gemv(int clear);
int debug_bounds_gemv_f16(int clear);
int debug_bounds_gemm(int clear);
cudaError_t launch_bounds_selftest(cudaStream_t s);
#endif

}  // namespace syn

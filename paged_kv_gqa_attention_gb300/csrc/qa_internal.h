// Internal interface between the C-ABI layer (qa_api.cu) and the kernel
// translation units.  Not installed, not exported.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "qa.h"

namespace qa {

// ---- decode (decode.cu)
// CTAs of the persistent split-K decode grid on `device` (one per SM).
int decode_grid_ctas(int device);
// Workspace bytes for the split-K partials.
size_t decode_workspace_bytes(int batch, int n_q_heads, int head_dim, int ctas);
// Largest batch the decode kernel accepts (its page prefix sums live in
// shared memory).
constexpr int kDecodeMaxBatch = 4096;
// The fused decode step: q is the pre-norm projection; the new token (pre-norm
// k, v) is normalised, rotated and appended at position seq_lens[b] - 1.
struct DecodeAppend {
    const void *k_new, *v_new;
    const float *q_gain, *k_gain;
    void *k_pages, *v_pages;  // the same pools, writable
    float rms_eps, rope_theta;
};
cudaError_t launch_decode(const void *q, const void *k_pages, const void *v_pages,
                          const int32_t *page_table, const int32_t *seq_lens, int batch, void *out,
                          const qa_attn_params &p, float scale, int ctas, cudaStream_t stream,
                          const DecodeAppend *app = nullptr);
unsigned int status_read_clear_decode(cudaStream_t stream, cudaError_t *err);
// one CTA whose bounded wait expires after limit_us (decode.cu's status word)
cudaError_t launch_bounded_wait_check(unsigned int limit_us, cudaStream_t stream);

// ---- prefill (prefill.cu): causal attention with the KV page write fused in
// n_past: cached positions per request (chunked prefill), or nullptr (none)
cudaError_t launch_prefill(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                           const int32_t *n_past, int batch, int total_tokens, const int32_t *page_table,
                           void *k_pages, void *v_pages, void *out, const qa_attn_params &p, float scale,
                           cudaStream_t stream);
unsigned int status_read_clear_prefill(cudaStream_t stream, cudaError_t *err);

// ---- decode append (append.cu): QK-norm + NEOX RoPE + page write of the new token
cudaError_t launch_append(const void *q, const void *k, const void *v, const float *q_gain, const float *k_gain,
                          float rms_eps, float rope_theta, const int32_t *page_table, const int32_t *seq_lens,
                          int batch, void *k_pages, void *v_pages, void *q_out, const qa_attn_params &p,
                          cudaStream_t stream);
unsigned int status_read_clear_append(cudaStream_t stream, cudaError_t *err);

// ---- window (window.cu)
// ld_qkv: row stride (elements) of q, k and v; 0 = packed (n_q_heads * head_dim)
// job_ctr: two zero words of device memory (jobs claimed dynamically, the
// kernel leaves them zero), or nullptr (fixed job order)
cudaError_t launch_window(const void *q, const void *k, const void *v, const int32_t *cu_windows,
                          int n_windows, int total_tokens, void *out, const qa_attn_params &p,
                          float scale, cudaStream_t stream, long long ld_qkv = 0, int *job_ctr = nullptr);
unsigned int status_read_clear_window(cudaStream_t stream, cudaError_t *err);

// ---- dense projections (gemm.cu): out = act(x W^T + bias) + res, bf16,
// row strides in elements (multiples of 8); act 0 none, 1 exact gelu
cudaError_t launch_gemm(const void *x, long long ldx, int M, int K, const void *w, int N, const void *bias, int act,
                        const void *res, long long ldr, void *out, long long ldc, cudaStream_t stream);
unsigned int status_read_clear_gemm(cudaStream_t stream, cudaError_t *err);

// ---- encoder layer (encoder.cu)
bool layer_norm_supported(int d);
// zero2: two int32 words the kernel sets to zero as well (nullptr: none)
cudaError_t launch_layer_norm(const void *x, int T, int d, const void *g, const void *b, float eps, void *y,
                              cudaStream_t stream, int *zero2 = nullptr);
// byte offsets of the layer's intermediates in the caller's workspace (ctr:
// the window attention's job counter)
struct EncoderWorkspace {
    size_t ctr, a, qkv, o, h, f, total;
};
EncoderWorkspace encoder_workspace_layout(long long T, int d, int d_ffn);
cudaError_t launch_encoder_layer(const void *x, const int32_t *cu_windows, int n_windows, int T, int d, int H,
                                 int d_ffn, const qa_encoder_weights &w, float eps, void *workspace, void *out,
                                 const qa_attn_params &p, cudaStream_t stream);

// ---- qa_api.cu
// Writes the thread-local qa_last_error() message.
void set_last_error(const char *msg);
// CTAs of the decode grid on the current device (0 when there is none).
int current_decode_ctas();
// Host checks of a decode call, everything but the workspace: the params
// (ABI range, scale, stable_metadata, shape), the tensor pointers, the batch
// and the alignments.  Sets qa_last_error() and returns INVALID_PARAMS on the
// first failure.
qa_status check_decode_call(const char *fn, const void *q, const void *k_pages, const void *v_pages,
                            const int32_t *page_table, const int32_t *seq_lens, int batch, const void *out,
                            const qa_attn_params *p);

}  // namespace qa

// C-ABI layer of libqa: argument validation, status codes, the thread-local
// last-error slot, and dispatch to the kernel launchers.  Conventions follow
// the qwenasr.cpp public ABI (qwenasr.cpp ARCHITECTURE.md, "Public API":
// status codes, thread-local qa_last_error, abi_version guarding struct
// growth; "ABI guarantee": only qa_* symbols exported).
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "qa.h"
#include "qa_internal.h"

#define QA_API extern "C" __attribute__((visibility("default")))

namespace {

thread_local char t_last_error[512] = "";

qa_status fail(qa_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return st;
}

void clear_error() { t_last_error[0] = '\0'; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// RoPE angles are reduced in fp32 with an exact first step for positions
// below 2^18 (sincos_pos_freq).
constexpr int kMaxRopePositions = 1 << 18;

qa_status check_common(const qa_attn_params *p, const char *fn) {
    if (!p) return fail(QA_STATUS_INVALID_PARAMS, "%s: params is NULL", fn);
    if (p->abi_version < QA_ABI_MIN_VERSION || p->abi_version > QA_ABI_VERSION)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: abi_version %d outside [%d, %d]", fn, p->abi_version,
                    QA_ABI_MIN_VERSION, QA_ABI_VERSION);
    if (!(p->scale >= 0.f) || !isfinite(p->scale))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: scale must be finite and >= 0 (0 = 1/sqrt(head_dim))", fn);
    if (p->abi_version >= 2 && (p->stable_metadata < 0 || p->stable_metadata > 2))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: stable_metadata %d outside [0, 2]", fn, p->stable_metadata);
    return QA_STATUS_OK;
}

float effective_scale(const qa_attn_params *p) {
    return p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)p->head_dim);
}

qa_status check_gqa(const qa_attn_params *p, const char *fn) {
    if (p->head_dim != 128)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: head_dim %d unsupported (128 only)", fn, p->head_dim);
    if (p->n_kv_heads < 1 || p->n_kv_heads > 8)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: n_kv_heads %d outside [1, 8]", fn, p->n_kv_heads);
    if (p->n_q_heads != p->n_kv_heads && p->n_q_heads != 2 * p->n_kv_heads)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: n_q_heads %d must be n_kv_heads or 2 * n_kv_heads (%d)", fn,
                    p->n_q_heads, p->n_kv_heads);
    if (p->page_size != 16)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: page_size %d unsupported (16 only)", fn, p->page_size);
    if (p->num_pages < 1 || p->max_pages_per_seq < 1)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: num_pages (%d) and max_pages_per_seq (%d) must be >= 1", fn,
                    p->num_pages, p->max_pages_per_seq);
    if ((long long)p->max_pages_per_seq * p->page_size > 0x7fffffffLL)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: max_pages_per_seq * page_size overflows int32", fn);
    return QA_STATUS_OK;
}

qa_status launch_result(cudaError_t e, const char *fn) {
    if (e != cudaSuccess) return fail(QA_STATUS_LAUNCH_FAILED, "%s: CUDA error %s", fn, cudaGetErrorString(e));
    return QA_STATUS_OK;
}

qa_status debug_status(unsigned int bits, cudaError_t e, const char *fn) {
    if (e != cudaSuccess) return fail(QA_STATUS_LAUNCH_FAILED, "%s: CUDA error %s", fn, cudaGetErrorString(e));
    if (bits)
        return fail(QA_STATUS_DEVICE_ERROR, "%s: device status 0x%x (%s%s%s%s)", fn, bits,
                    bits & QA_DEVICE_BAD_PAGE ? "bad page id " : "", bits & QA_DEVICE_BAD_LENGTH ? "bad length " : "",
                    bits & QA_DEVICE_BAD_SEGMENTS ? "bad segments " : "", bits & QA_DEVICE_TIMEOUT ? "timeout" : "");
    return QA_STATUS_OK;
}

}  // namespace

namespace qa {

int current_decode_ctas() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return decode_grid_ctas(dev);
    if (cache[dev] == 0) cache[dev] = decode_grid_ctas(dev);
    return cache[dev];
}

qa_status check_decode_call(const char *fn, const void *q, const void *k_pages, const void *v_pages,
                            const int32_t *page_table, const int32_t *seq_lens, int batch, const void *out,
                            const qa_attn_params *p) {
    qa_status st = check_common(p, fn);
    if (st != QA_STATUS_OK) return st;
    if ((st = check_gqa(p, fn)) != QA_STATUS_OK) return st;
    if (!q || !k_pages || !v_pages || !page_table || !seq_lens || !out)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: NULL tensor pointer", fn);
    if (batch < 1 || batch > kDecodeMaxBatch)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: batch %d outside [1, %d]", fn, batch, kDecodeMaxBatch);
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(page_table, 4) || !aligned(seq_lens, 4))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: tensors must be 16-byte aligned (int32 arrays 4-byte)", fn);
    return QA_STATUS_OK;
}

}  // namespace qa

QA_API qa_attn_params qa_attn_default_params(void) {
    qa_attn_params p;
    p.abi_version = QA_ABI_VERSION;
    p.n_q_heads = 16;
    p.n_kv_heads = 8;
    p.head_dim = 128;
    p.page_size = 16;
    p.num_pages = 0;
    p.max_pages_per_seq = 0;
    p.scale = 0.f;
    p.stream = nullptr;
    p.workspace = nullptr;
    p.workspace_bytes = 0;
    p.debug_checks = 0;
    p.stable_metadata = 0;
    return p;
}

QA_API size_t qa_decode_workspace_size(int batch, int max_seq_len, const qa_attn_params *p) {
    clear_error();
    if (check_common(p, "qa_decode_workspace_size") != QA_STATUS_OK) return 0;
    if (check_gqa(p, "qa_decode_workspace_size") != QA_STATUS_OK) return 0;
    if (batch < 1 || batch > qa::kDecodeMaxBatch) {
        fail(QA_STATUS_INVALID_PARAMS, "qa_decode_workspace_size: batch %d outside [1, %d]", batch, qa::kDecodeMaxBatch);
        return 0;
    }
    if (max_seq_len < 0 || (long long)max_seq_len > (long long)p->max_pages_per_seq * p->page_size) {
        fail(QA_STATUS_INVALID_PARAMS, "qa_decode_workspace_size: max_seq_len %d outside [0, max_pages_per_seq * page_size]",
             max_seq_len);
        return 0;
    }
    const int ctas = qa::current_decode_ctas();
    if (ctas <= 0) {
        fail(QA_STATUS_LAUNCH_FAILED, "qa_decode_workspace_size: no CUDA device");
        return 0;
    }
    return qa::decode_workspace_bytes(batch, p->n_q_heads, p->head_dim, ctas);
}

namespace {

// Shared by qa_decode_attn and qa_decode_step (app != nullptr).
qa_status decode_entry(const char *fn, const void *q, const void *k_pages, const void *v_pages,
                       const int32_t *page_table, const int32_t *seq_lens, int batch, void *out,
                       const qa_attn_params *p, const qa::DecodeAppend *app) {
    qa_status st = qa::check_decode_call(fn, q, k_pages, v_pages, page_table, seq_lens, batch, out, p);
    if (st != QA_STATUS_OK) return st;
    const int ctas = qa::current_decode_ctas();
    if (ctas <= 0) return fail(QA_STATUS_LAUNCH_FAILED, "%s: no CUDA device", fn);
    const size_t need = qa::decode_workspace_bytes(batch, p->n_q_heads, p->head_dim, ctas);
    if (!p->workspace || p->workspace_bytes < need || !aligned(p->workspace, 256))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: workspace must be >= %zu bytes and 256-byte aligned (got %zu)", fn,
                    need, p->workspace_bytes);
    cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
    st = launch_result(qa::launch_decode(q, k_pages, v_pages, page_table, seq_lens, batch, out, *p,
                                         effective_scale(p), ctas, stream, app),
                       fn);
    if (st != QA_STATUS_OK || !p->debug_checks) return st;
    cudaError_t e;
    const unsigned int bits = qa::status_read_clear_decode(stream, &e);
    return debug_status(bits, e, fn);
}

}  // namespace

QA_API qa_status qa_decode_attn(const void *q, const void *k_pages, const void *v_pages, const int32_t *page_table,
                                const int32_t *seq_lens, int batch, void *out, const qa_attn_params *p) {
    clear_error();
    return decode_entry("qa_decode_attn", q, k_pages, v_pages, page_table, seq_lens, batch, out, p, nullptr);
}

QA_API qa_status qa_decode_step(const void *q, const void *k, const void *v, const float *q_gain, const float *k_gain,
                                float rms_eps, float rope_theta, void *k_pages, void *v_pages,
                                const int32_t *page_table, const int32_t *seq_lens, int batch, void *out,
                                const qa_attn_params *p) {
    const char *fn = "qa_decode_step";
    clear_error();
    if (!(rms_eps > 0.f) || !isfinite(rms_eps))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: rms_eps must be finite and > 0", fn);
    if (!(rope_theta > 0.f) || !isfinite(rope_theta))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: rope_theta must be finite and > 0", fn);
    if (p && (long long)p->max_pages_per_seq * p->page_size > kMaxRopePositions)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: positions up to %d supported (max_pages_per_seq * page_size = %lld)",
                    fn, kMaxRopePositions, (long long)p->max_pages_per_seq * p->page_size);
    if (!k || !v || !q_gain || !k_gain) return fail(QA_STATUS_INVALID_PARAMS, "%s: NULL pointer", fn);
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(q_gain, 16) || !aligned(k_gain, 16))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: k, v and the gains must be 16-byte aligned", fn);
    qa::DecodeAppend app{k, v, q_gain, k_gain, k_pages, v_pages, rms_eps, rope_theta};
    return decode_entry(fn, q, k_pages, v_pages, page_table, seq_lens, batch, out, p, &app);
}

namespace {

// Shared by qa_prefill_attn (n_past == nullptr) and qa_prefill_chunk_attn.
qa_status prefill_entry(const char *fn, const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                        const int32_t *n_past, int batch, int total_tokens, const int32_t *page_table,
                        void *k_pages, void *v_pages, void *out, const qa_attn_params *p) {
    qa_status st = check_common(p, fn);
    if (st != QA_STATUS_OK) return st;
    if ((st = check_gqa(p, fn)) != QA_STATUS_OK) return st;
    if (batch < 1) return fail(QA_STATUS_INVALID_PARAMS, "%s: batch %d < 1", fn, batch);
    if (total_tokens < 0) return fail(QA_STATUS_INVALID_PARAMS, "%s: total_tokens %d < 0", fn, total_tokens);
    if ((long long)total_tokens * p->n_q_heads * p->head_dim > (1LL << 40))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: total_tokens %d too large", fn, total_tokens);
    if ((long long)p->num_pages * p->page_size > 0x7fffffffLL)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: num_pages * page_size overflows int32", fn);
    if (!q || !k || !v || !cu_seqlens || !page_table || !k_pages || !v_pages || !out)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: NULL tensor pointer", fn);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(k_pages, 16) ||
        !aligned(v_pages, 16) || !aligned(cu_seqlens, 4) || !aligned(page_table, 4) || !aligned(n_past, 4))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: tensors must be 16-byte aligned (int32 arrays 4-byte)", fn);
    cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
    st = launch_result(qa::launch_prefill(q, k, v, cu_seqlens, n_past, batch, total_tokens, page_table, k_pages,
                                          v_pages, out, *p, effective_scale(p), stream),
                       fn);
    if (st != QA_STATUS_OK || !p->debug_checks) return st;
    cudaError_t e;
    const unsigned int bits = qa::status_read_clear_prefill(stream, &e);
    return debug_status(bits, e, fn);
}

}  // namespace

QA_API qa_status qa_prefill_attn(const void *q, const void *k, const void *v, const int32_t *cu_seqlens, int batch,
                                 int total_tokens, const int32_t *page_table, void *k_pages, void *v_pages, void *out,
                                 const qa_attn_params *p) {
    clear_error();
    return prefill_entry("qa_prefill_attn", q, k, v, cu_seqlens, nullptr, batch, total_tokens, page_table, k_pages,
                         v_pages, out, p);
}

QA_API qa_status qa_prefill_chunk_attn(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                                       const int32_t *n_past, int batch, int total_tokens,
                                       const int32_t *page_table, void *k_pages, void *v_pages, void *out,
                                       const qa_attn_params *p) {
    clear_error();
    if (!n_past) return fail(QA_STATUS_INVALID_PARAMS, "qa_prefill_chunk_attn: n_past is NULL");
    return prefill_entry("qa_prefill_chunk_attn", q, k, v, cu_seqlens, n_past, batch, total_tokens, page_table,
                         k_pages, v_pages, out, p);
}

QA_API qa_status qa_decode_append(const void *q, const void *k, const void *v, const float *q_gain,
                                  const float *k_gain, float rms_eps, float rope_theta, const int32_t *page_table,
                                  const int32_t *seq_lens, int batch, void *k_pages, void *v_pages, void *q_out,
                                  const qa_attn_params *p) {
    const char *fn = "qa_decode_append";
    clear_error();
    qa_status st = check_common(p, fn);
    if (st != QA_STATUS_OK) return st;
    if ((st = check_gqa(p, fn)) != QA_STATUS_OK) return st;
    if (!(rms_eps > 0.f) || !isfinite(rms_eps))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: rms_eps must be finite and > 0", fn);
    if (!(rope_theta > 0.f) || !isfinite(rope_theta))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: rope_theta must be finite and > 0", fn);
    if ((long long)p->max_pages_per_seq * p->page_size > kMaxRopePositions)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: positions up to %d supported (max_pages_per_seq * page_size = %lld)",
                    fn, kMaxRopePositions, (long long)p->max_pages_per_seq * p->page_size);
    if (batch < 1) return fail(QA_STATUS_INVALID_PARAMS, "%s: batch %d < 1", fn, batch);
    if (!q || !k || !v || !q_gain || !k_gain || !page_table || !seq_lens || !k_pages || !v_pages || !q_out)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: NULL pointer", fn);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q_out, 16) || !aligned(k_pages, 16) ||
        !aligned(v_pages, 16) || !aligned(q_gain, 8) || !aligned(k_gain, 8) || !aligned(page_table, 4) ||
        !aligned(seq_lens, 4))
        return fail(QA_STATUS_INVALID_PARAMS,
                    "%s: tensors must be 16-byte aligned (gains 8-byte, int32 arrays 4-byte)", fn);
    cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
    st = launch_result(qa::launch_append(q, k, v, q_gain, k_gain, rms_eps, rope_theta, page_table, seq_lens, batch,
                                         k_pages, v_pages, q_out, *p, stream),
                       fn);
    if (st != QA_STATUS_OK || !p->debug_checks) return st;
    cudaError_t e;
    const unsigned int bits = qa::status_read_clear_append(stream, &e);
    return debug_status(bits, e, fn);
}

QA_API qa_status qa_window_attn(const void *q, const void *k, const void *v, const int32_t *cu_windows, int n_windows,
                                int total_tokens, void *out, const qa_attn_params *p) {
    const char *fn = "qa_window_attn";
    clear_error();
    qa_status st = check_common(p, fn);
    if (st != QA_STATUS_OK) return st;
    if (p->head_dim != 64 && p->head_dim != 128)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: head_dim %d unsupported (64 or 128)", fn, p->head_dim);
    if (p->n_q_heads < 1 || p->n_kv_heads != p->n_q_heads)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: n_q_heads (%d) must equal n_kv_heads (%d) and be >= 1", fn,
                    p->n_q_heads, p->n_kv_heads);
    if (n_windows < 1) return fail(QA_STATUS_INVALID_PARAMS, "%s: n_windows %d < 1", fn, n_windows);
    if (total_tokens < 0) return fail(QA_STATUS_INVALID_PARAMS, "%s: total_tokens %d < 0", fn, total_tokens);
    if ((long long)total_tokens * p->n_q_heads * p->head_dim > (1LL << 40))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: total_tokens %d too large", fn, total_tokens);
    if (!q || !k || !v || !cu_windows || !out) return fail(QA_STATUS_INVALID_PARAMS, "%s: NULL tensor pointer", fn);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(cu_windows, 4))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: tensors must be 16-byte aligned (int32 arrays 4-byte)", fn);
    int *job_ctr = nullptr;
    if (p->workspace) {
        if (p->workspace_bytes < qa_window_workspace_size() || !aligned(p->workspace, 4))
            return fail(QA_STATUS_INVALID_PARAMS, "%s: workspace of %zu bytes (needs %zu, 4-byte aligned)", fn,
                        p->workspace_bytes, qa_window_workspace_size());
        job_ctr = static_cast<int *>(p->workspace);
    }
    cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
    st = launch_result(qa::launch_window(q, k, v, cu_windows, n_windows, total_tokens, out, *p, effective_scale(p),
                                         stream, 0, job_ctr),
                       fn);
    if (st != QA_STATUS_OK || !p->debug_checks) return st;
    cudaError_t e;
    const unsigned int bits = qa::status_read_clear_window(stream, &e);
    return debug_status(bits, e, fn);
}

QA_API size_t qa_window_workspace_size(void) { return 256; }

QA_API int qa_window_plan(const int32_t *token_counts, int n_requests, int window_tokens, int32_t *cu_windows,
                          int capacity) {
    clear_error();
    if (n_requests < 0 || (n_requests > 0 && !token_counts) || !cu_windows || capacity < 1) {
        fail(QA_STATUS_INVALID_PARAMS, "qa_window_plan: bad arguments");
        return -1;
    }
    // window_aftercnn = conv_out(chunk_mel) * window_chunks = 13 * 8 = 104
    const int w = window_tokens > 0 ? window_tokens : 104;
    long long offset = 0;
    int n = 0;
    cu_windows[0] = 0;
    for (int r = 0; r < n_requests; ++r) {
        const int count = token_counts[r];
        if (count < 0) {
            fail(QA_STATUS_INVALID_PARAMS, "qa_window_plan: token_counts[%d] = %d < 0", r, count);
            return -1;
        }
        for (int start = 0; start < count; start += w) {
            const int len = count - start < w ? count - start : w;
            offset += len;
            if (offset > 0x7fffffffLL) {
                fail(QA_STATUS_INVALID_PARAMS, "qa_window_plan: total tokens overflow int32");
                return -1;
            }
            if (n + 2 > capacity) {
                fail(QA_STATUS_INVALID_PARAMS, "qa_window_plan: capacity %d too small", capacity);
                return -1;
            }
            cu_windows[++n] = (int32_t)offset;
        }
    }
    return n;
}

QA_API size_t qa_encoder_workspace_size(int total_tokens, int d_model, int d_ffn) {
    clear_error();
    if (total_tokens < 0 || d_model < 1 || d_ffn < 1) {
        fail(QA_STATUS_INVALID_PARAMS, "qa_encoder_workspace_size: bad sizes");
        return 0;
    }
    return qa::encoder_workspace_layout(total_tokens, d_model, d_ffn).total;
}

QA_API qa_status qa_encoder_layer(const void *x, const int32_t *cu_windows, int n_windows, int total_tokens,
                                  int d_model, int n_heads, int d_ffn, const qa_encoder_weights *w, float ln_eps,
                                  void *out, const qa_attn_params *p) {
    const char *fn = "qa_encoder_layer";
    clear_error();
    qa_status st = check_common(p, fn);
    if (st != QA_STATUS_OK) return st;
    if (!qa::layer_norm_supported(d_model))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: d_model %d unsupported (a multiple of 128 up to 2048)", fn,
                    d_model);
    if (n_heads < 1 || d_model % n_heads || (d_model / n_heads != 64 && d_model / n_heads != 128))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: d_model / n_heads must be 64 or 128 (d_model %d, n_heads %d)", fn,
                    d_model, n_heads);
    if (d_ffn < 8 || d_ffn % 8) return fail(QA_STATUS_INVALID_PARAMS, "%s: d_ffn %d must be a multiple of 8", fn, d_ffn);
    if (n_windows < 1) return fail(QA_STATUS_INVALID_PARAMS, "%s: n_windows %d < 1", fn, n_windows);
    if (total_tokens < 0) return fail(QA_STATUS_INVALID_PARAMS, "%s: total_tokens %d < 0", fn, total_tokens);
    if (!(ln_eps >= 0.f) || !isfinite(ln_eps))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: ln_eps must be finite and >= 0", fn);
    if (!x || !cu_windows || !out || !w) return fail(QA_STATUS_INVALID_PARAMS, "%s: NULL pointer", fn);
    const void *wp[12] = {w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_o, w->b_o,
                          w->ln2_g, w->ln2_b, w->w_fc1, w->b_fc1, w->w_fc2, w->b_fc2};
    for (const void *q : wp) {
        if (!q) return fail(QA_STATUS_INVALID_PARAMS, "%s: NULL weight pointer", fn);
        if (!aligned(q, 16)) return fail(QA_STATUS_INVALID_PARAMS, "%s: weights must be 16-byte aligned", fn);
    }
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(cu_windows, 4))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: x and out must be 16-byte aligned (cu_windows 4-byte)", fn);
    if (x == out) return fail(QA_STATUS_INVALID_PARAMS, "%s: out may not alias x", fn);
    const size_t need = qa::encoder_workspace_layout(total_tokens, d_model, d_ffn).total;
    if (!p->workspace || p->workspace_bytes < need || !aligned(p->workspace, 256))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: workspace must be >= %zu bytes and 256-byte aligned (got %zu)", fn,
                    need, p->workspace_bytes);
    cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
    st = launch_result(qa::launch_encoder_layer(x, cu_windows, n_windows, total_tokens, d_model, n_heads, d_ffn, *w,
                                                ln_eps, p->workspace, out, *p, stream),
                       fn);
    if (st != QA_STATUS_OK || !p->debug_checks) return st;
    cudaError_t e[2];
    const unsigned int bits = qa::status_read_clear_window(stream, &e[0]) | qa::status_read_clear_gemm(stream, &e[1]);
    return debug_status(bits, e[0] != cudaSuccess ? e[0] : e[1], fn);
}

QA_API qa_status qa_linear(const void *x, int m, int k, const void *w, int n, const void *bias, int act,
                           const void *residual, void *out, const qa_attn_params *p) {
    const char *fn = "qa_linear";
    clear_error();
    qa_status st = check_common(p, fn);
    if (st != QA_STATUS_OK) return st;
    if (m < 0 || k < 8 || k % 8 || n < 8 || n % 8)
        return fail(QA_STATUS_INVALID_PARAMS, "%s: m %d >= 0, k %d and n %d multiples of 8 required", fn, m, k, n);
    if (act != 0 && act != 1) return fail(QA_STATUS_INVALID_PARAMS, "%s: act %d must be 0 or 1", fn, act);
    if (!x || !w || !out) return fail(QA_STATUS_INVALID_PARAMS, "%s: NULL pointer", fn);
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(out, 16) || !aligned(bias, 16) || !aligned(residual, 16))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: tensors must be 16-byte aligned", fn);
    cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
    st = launch_result(qa::launch_gemm(x, k, m, k, w, n, bias, act, residual, n, out, n, stream), fn);
    if (st != QA_STATUS_OK || !p->debug_checks) return st;
    cudaError_t e;
    const unsigned int bits = qa::status_read_clear_gemm(stream, &e);
    return debug_status(bits, e, fn);
}

QA_API qa_status qa_layer_norm(const void *x, int t, int d, const void *gain, const void *bias, float eps, void *y,
                               const qa_attn_params *p) {
    const char *fn = "qa_layer_norm";
    clear_error();
    qa_status st = check_common(p, fn);
    if (st != QA_STATUS_OK) return st;
    if (t < 0 || !qa::layer_norm_supported(d))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: t %d >= 0 and d %d a multiple of 128 up to 2048 required", fn, t,
                    d);
    if (!(eps >= 0.f) || !isfinite(eps)) return fail(QA_STATUS_INVALID_PARAMS, "%s: eps must be finite and >= 0", fn);
    if (!x || !gain || !bias || !y) return fail(QA_STATUS_INVALID_PARAMS, "%s: NULL pointer", fn);
    if (!aligned(x, 16) || !aligned(gain, 16) || !aligned(bias, 16) || !aligned(y, 16))
        return fail(QA_STATUS_INVALID_PARAMS, "%s: tensors must be 16-byte aligned", fn);
    cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
    st = launch_result(qa::launch_layer_norm(x, t, d, gain, bias, eps, y, stream), fn);
    if (st != QA_STATUS_OK || !p->debug_checks) return st;
    cudaError_t e = cudaStreamSynchronize(stream);
    return launch_result(e, fn);
}

QA_API int qa_device_status(void *stream) {
    clear_error();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e[5];
    const unsigned int bits = qa::status_read_clear_decode(s, &e[0]) | qa::status_read_clear_prefill(s, &e[1]) |
                              qa::status_read_clear_window(s, &e[2]) | qa::status_read_clear_append(s, &e[3]) |
                              qa::status_read_clear_gemm(s, &e[4]);
    for (cudaError_t ei : e)
        if (ei != cudaSuccess) {
            fail(QA_STATUS_LAUNCH_FAILED, "qa_device_status: CUDA error %s", cudaGetErrorString(ei));
            return -1;
        }
    return (int)bits;
}

QA_API qa_status qa_check_bounded_wait(unsigned int limit_us, void *stream) {
    clear_error();
    if (limit_us < 1 || limit_us > 1000000u)
        return fail(QA_STATUS_INVALID_PARAMS, "qa_check_bounded_wait: limit_us %u outside [1, 1000000]", limit_us);
    const cudaError_t e = qa::launch_bounded_wait_check(limit_us, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(QA_STATUS_LAUNCH_FAILED, "qa_check_bounded_wait: CUDA error %s", cudaGetErrorString(e));
    return QA_STATUS_OK;
}

QA_API const char *qa_last_error(void) { return t_last_error; }

QA_API const char *qa_version(void) {
    static char v[64];
    snprintf(v, sizeof v, "qa-attn 0.1.0 abi %d", QA_ABI_VERSION);
    return v;
}

namespace qa {
// Lets entry points defined in other translation units report through the
// same thread-local qa_last_error() slot.
void set_last_error(const char *msg) { snprintf(t_last_error, sizeof t_last_error, "%s", msg); }
}  // namespace qa

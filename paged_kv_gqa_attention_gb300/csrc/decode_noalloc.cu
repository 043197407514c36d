// qa_decode_attn_noalloc: the paged decode for callers that cannot allocate
// device memory.
//
// qa_decode_attn needs caller-provided scratch (the split-K partial results).
// Some callers cannot obtain it: a plugin whose host application owns every
// device allocation and forbids cudaMalloc, a real-time audio path that may
// not block on (or fail in) an allocator, or a C program that links only this
// library and has no allocator of its own.  This entry point runs the same
// decode kernels with their scratch in a fixed array compiled into the
// library instead, so the caller passes only inputs and outputs.
//
// Costs and limits: the array (kScratchBytes, 4 MiB) is reserved on every GPU
// that loads the library, for the life of the process.  A call whose batch
// needs more scratch than that is rejected before any launch.  All calls on a
// device share the one array: two calls whose kernels overlap on the GPU
// (different streams, or different host threads, without ordering between
// them) race on it and give wrong results; calls ordered on one stream are
// fine.  The array keeps whatever the last call left in it.  The only part
// that must start at zero is the block of per-request arrival counters at
// its head (a fixed-size region whatever the batch): the loader zero-fills
// the array and every call leaves the counters it used at zero again; the
// partial results behind them are always written before they are read.
//
// Set-up: the device address of the array is looked up (cudaGetSymbolAddress)
// on the first call made with each device current and cached per device, so
// that first call should be made before any CUDA stream capture begins.
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "qa.h"
#include "qa_internal.h"

#define QA_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kScratchBytes = (size_t)4 << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

qa_status reject(qa_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
qa_status reject(qa_status st, const char *fmt, ...) {
    char msg[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    qa::set_last_error(msg);
    return st;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Device address of the scratch array on the current device (set up once per
// device).  Returns nullptr and fills *err on failure.
void *scratch_on_current_device(cudaError_t *err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (*err != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

QA_API qa_status qa_decode_attn_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                        const int32_t *page_table, const int32_t *seq_lens, int batch, void *out,
                                        const qa_attn_params *p) {
    const char *fn = "qa_decode_attn_noalloc";
    qa::set_last_error("");
    if (!p) return reject(QA_STATUS_INVALID_PARAMS, "%s: params is NULL", fn);
    if (p->abi_version < QA_ABI_MIN_VERSION || p->abi_version > QA_ABI_VERSION)
        return reject(QA_STATUS_INVALID_PARAMS, "%s: abi_version %d outside [%d, %d]", fn, p->abi_version,
                      QA_ABI_MIN_VERSION, QA_ABI_VERSION);
    if (!(p->scale >= 0.f) || !isfinite(p->scale))
        return reject(QA_STATUS_INVALID_PARAMS, "%s: scale must be finite and >= 0 (0 = 1/sqrt(head_dim))", fn);
    if (p->head_dim != 128 || p->page_size != 16 || p->n_kv_heads < 1 || p->n_kv_heads > 8 ||
        (p->n_q_heads != p->n_kv_heads && p->n_q_heads != 2 * p->n_kv_heads))
        return reject(QA_STATUS_INVALID_PARAMS,
                      "%s: unsupported shape (head_dim 128, page_size 16, n_kv_heads 1..8, n_q_heads = 1 or 2 x "
                      "n_kv_heads)",
                      fn);
    if (p->num_pages < 1 || p->max_pages_per_seq < 1 || (long long)p->max_pages_per_seq * p->page_size > 0x7fffffffLL)
        return reject(QA_STATUS_INVALID_PARAMS, "%s: num_pages and max_pages_per_seq must be >= 1 (and fit int32)", fn);
    if (!q || !k_pages || !v_pages || !page_table || !seq_lens || !out)
        return reject(QA_STATUS_INVALID_PARAMS, "%s: NULL tensor pointer", fn);
    if (batch < 1 || batch > qa::kDecodeMaxBatch)
        return reject(QA_STATUS_INVALID_PARAMS, "%s: batch %d outside [1, %d]", fn, batch, qa::kDecodeMaxBatch);
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(page_table, 4) || !aligned(seq_lens, 4))
        return reject(QA_STATUS_INVALID_PARAMS, "%s: tensors must be 16-byte aligned (int32 arrays 4-byte)", fn);

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return reject(QA_STATUS_LAUNCH_FAILED, "%s: no CUDA device", fn);
    const int ctas = qa::decode_grid_ctas(dev);
    if (ctas <= 0) return reject(QA_STATUS_LAUNCH_FAILED, "%s: no CUDA device", fn);
    const size_t need = qa::decode_workspace_bytes(batch, p->n_q_heads, p->head_dim, ctas);
    if (need > kScratchBytes)
        return reject(QA_STATUS_INVALID_PARAMS,
                      "%s: batch %d with %d query heads needs %zu bytes of scratch; the built-in array holds %zu "
                      "(use qa_decode_attn with a caller workspace for larger batches)",
                      fn, batch, p->n_q_heads, need, kScratchBytes);

    cudaError_t e;
    void *scratch = scratch_on_current_device(&e);
    if (!scratch)
        return reject(QA_STATUS_LAUNCH_FAILED, "%s: cannot find the scratch array's device address: %s", fn,
                      cudaGetErrorString(e));

    qa_attn_params local = *p;
    local.workspace = scratch;
    local.workspace_bytes = kScratchBytes;
    const float scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)p->head_dim);
    cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
    e = qa::launch_decode(q, k_pages, v_pages, page_table, seq_lens, batch, out, local, scale, ctas, stream);
    if (e != cudaSuccess) return reject(QA_STATUS_LAUNCH_FAILED, "%s: CUDA error %s", fn, cudaGetErrorString(e));
    if (!p->debug_checks) return QA_STATUS_OK;
    const unsigned int bits = qa::status_read_clear_decode(stream, &e);
    if (e != cudaSuccess) return reject(QA_STATUS_LAUNCH_FAILED, "%s: CUDA error %s", fn, cudaGetErrorString(e));
    if (bits) return reject(QA_STATUS_DEVICE_ERROR, "%s: device status 0x%x", fn, bits);
    return QA_STATUS_OK;
}

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
// Set-up: every call looks up the device address of the array on the current
// device (cudaGetSymbolAddress) and passes it to the kernel.  Host code cannot
// name the array directly (its host-side name is only a stand-in), and the
// address is not cached: it belongs to the module loaded in the current
// context, which a cudaDeviceReset replaces.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "qa.h"
#include "qa_internal.h"

#define QA_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kScratchBytes = (size_t)4 << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

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

}  // namespace

QA_API qa_status qa_decode_attn_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                        const int32_t *page_table, const int32_t *seq_lens, int batch, void *out,
                                        const qa_attn_params *p) {
    const char *fn = "qa_decode_attn_noalloc";
    qa::set_last_error("");
    // the same checks as qa_decode_attn, minus its workspace
    const qa_status st = qa::check_decode_call(fn, q, k_pages, v_pages, page_table, seq_lens, batch, out, p);
    if (st != QA_STATUS_OK) return st;
    const int ctas = qa::current_decode_ctas();
    if (ctas <= 0) return reject(QA_STATUS_LAUNCH_FAILED, "%s: no CUDA device", fn);
    const size_t need = qa::decode_workspace_bytes(batch, p->n_q_heads, p->head_dim, ctas);
    if (need > kScratchBytes)
        return reject(QA_STATUS_INVALID_PARAMS,
                      "%s: batch %d with %d query heads needs %zu bytes of scratch; the built-in array holds %zu "
                      "(use qa_decode_attn with a caller workspace for larger batches)",
                      fn, batch, p->n_q_heads, need, kScratchBytes);

    void *scratch = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&scratch, g_decode_scratch);
    if (e != cudaSuccess || !scratch)
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

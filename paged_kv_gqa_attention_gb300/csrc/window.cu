// Windowed bidirectional encoder attention over a packed sequence.
//
// qwenasr.cpp ARCHITECTURE.md, "Windowed audio tower": the encoder attends
// under a block-diagonal mask over windows of 104 tokens; attention is plain
// bidirectional MHA scaled by 1/sqrt(head_dim).  M* "Speech recognition:
// Whisper and Qwen3-ASR", "Graph": one packed forward per batch with one
// segment per window of every request.  Row t of window w attends over every
// row of w and nothing else.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "qa_internal.h"
#include "row_attn.cuh"

namespace qa {
namespace {
__device__ unsigned int g_status;
}  // namespace

cudaError_t launch_window(const void *q, const void *k, const void *v, const int32_t *cu_windows,
                          int n_windows, int total_tokens, void *out, const qa_attn_params &p,
                          float scale, cudaStream_t stream) {
    if (total_tokens == 0) return cudaSuccess;
    RowAttnArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.k = static_cast<const uint16_t *>(k);
    a.v = static_cast<const uint16_t *>(v);
    a.cu = cu_windows;
    a.out = static_cast<uint16_t *>(out);
    a.n_seg = n_windows;
    a.total = total_tokens;
    a.hkv = p.n_kv_heads;
    a.scale_log2 = scale * kLog2e;
    unsigned int *status = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status);
    if (e != cudaSuccess) return e;
    const long long warps = (long long)total_tokens * a.hkv;
    const int blocks = (int)((warps + 7) / 8);
    if (p.head_dim == 64)
        row_attn_kernel<64, 1, false><<<blocks, 256, 0, stream>>>(a, status);
    else
        row_attn_kernel<128, 1, false><<<blocks, 256, 0, stream>>>(a, status);
    return cudaGetLastError();
}

unsigned int status_read_clear_window(cudaStream_t stream, cudaError_t *err) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status, sizeof v, 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && v) e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (err) *err = e;
    return v;
}

}  // namespace qa

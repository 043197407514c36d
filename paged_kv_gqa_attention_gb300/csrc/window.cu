// Windowed bidirectional encoder attention over a packed sequence.
//
// qwenasr.cpp ARCHITECTURE.md, "Windowed audio tower": the encoder attends
// under a block-diagonal mask over windows of 104 tokens; attention is plain
// bidirectional MHA scaled by 1/sqrt(head_dim).  M* "Speech recognition:
// Whisper and Qwen3-ASR", "Graph": one packed forward per batch with one
// segment per window of every request.  Row t of window w attends over every
// row of w and nothing else.  Runs on the tensor cores (attn_tc.cuh,
// window_tc_kernel): a persistent grid of four CTAs per SM (two for head_dim
// 128) walks the (window, head) jobs -- in a fixed order, or claimed one at a
// time from a job counter when the caller gives one; a 104-token window is
// one 128-row tile, longer windows loop over query and key tiles.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "qa_internal.h"
#include "attn_tc.cuh"
#include "tmap.h"

namespace qa {
namespace {
__device__ unsigned int g_status;
}  // namespace

cudaError_t launch_window(const void *q, const void *k, const void *v, const int32_t *cu_windows,
                          int n_windows, int total_tokens, void *out, const qa_attn_params &p,
                          float scale, cudaStream_t stream, long long ld_qkv, int *job_ctr) {
    if (total_tokens == 0) return cudaSuccess;
    if (p.n_q_heads > 65535) return cudaErrorInvalidValue;
    CUtensorMap tq, tk, tv, tout;
    // q, k and v may be column blocks of one wider row (ld_qkv elements apart)
    if (!make_rows_tmap(&tq, q, p.head_dim, p.n_q_heads, total_tokens, 128, ld_qkv) ||
        !make_rows_tmap(&tk, k, p.head_dim, p.n_kv_heads, total_tokens, 128, ld_qkv) ||
        !make_rows_tmap(&tv, v, p.head_dim, p.n_kv_heads, total_tokens, 128, ld_qkv))
        return cudaErrorInvalidValue;
    // the output is written in kOutBoxRows-row (32-row) TMA boxes (store_rows_tma)
    if (!make_rows_tmap(&tout, out, p.head_dim, p.n_q_heads, total_tokens, kOutBoxRows)) return cudaErrorInvalidValue;
    AttnTcArgs a{};
    a.cu = cu_windows;
    a.out = static_cast<uint16_t *>(out);
    a.n_seg = n_windows;
    a.total = total_tokens;
    a.hq = p.n_q_heads;
    a.scale_log2 = scale * kLog2e;
    a.job_ctr = job_ctr;
    unsigned int *status = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status);
    if (e != cudaSuccess) return e;
    // persistent grid: as many CTAs as fit on the GPU at once, at most one per job
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long n_jobs = (long long)n_windows * p.n_q_heads;
    if (n_jobs > 0x7fffffffLL) return cudaErrorInvalidValue;
    // CTAs per SM as the launch bounds size them (registers and shared memory
    // both fit: 4 x 49 KiB for head_dim 64, 2 x 97 KiB for 128); the
    // occupancy query under-reports for these kernels, so it is not used.
    // Extra CTAs would only queue: no CTA waits on another.
    auto launch = [&](auto kernel, uint32_t smem, int per_sm) -> cudaError_t {
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   (int)cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        const long long ctas = std::min<long long>(n_jobs, (long long)sms * per_sm);
        // a programmatic dependent of the kernel before it on the stream (it
        // waits for that kernel before it reads anything)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ctas);
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, tout, a, status);
    };
    if (p.head_dim == 64)
        e = launch(window_tc_kernel<64>, AttnTcLayout<64>::kSmem, 4);
    else
        e = launch(window_tc_kernel<128>, AttnTcLayout<128>::kSmem, 2);
    if (e != cudaSuccess) return e;
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

// Ragged causal prefill: the causal attention with the KV page write fused in.
//
// Page write (qwenasr.cpp ARCHITECTURE.md, "Qwen3 Thinker decoder": prefill
// rewinds the cache and writes the fresh K/V of the whole prompt span at
// [n_past, n_past + T) with n_past = 0): row i of request r is copied bit for
// bit to slot i % 16 of page page_table[r][i / 16], for K and V.  The jobs of
// query tile t for the two query heads of a KV head write the rows of tile t
// from their diagonal K/V tile, already in shared memory for the attention
// (the even head the K rows, the odd one the V rows; whole pages by TMA
// stores), so the prompt's K and V are read from HBM once for both.
//
// Attention: row i of request r attends over rows j <= i of the same request
// (same section: attend over [0, n_past + T)), GQA group h / 2, from the
// packed k and v, on the tensor cores (attn_tc.cuh, prefill_tc_kernel): one
// CTA per (128-row query tile, request, query head), longest jobs launched
// first, each over its causal key tiles 0..tile; the two query heads of a KV
// head are adjacent in launch order, so their K/V tiles come from L2 the
// second time.
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

cudaError_t launch_prefill(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                           const int32_t *n_past, int batch, int total_tokens, const int32_t *page_table,
                           void *k_pages, void *v_pages, void *out, const qa_attn_params &p, float scale,
                           cudaStream_t stream) {
    if (total_tokens == 0) return cudaSuccess;
    if (batch > 65535) return cudaErrorInvalidValue;
    CUtensorMap tq, tk, tv, tkp, tvp;
    const long long pool_rows = (long long)p.num_pages * p.page_size;
    if (!make_rows_tmap(&tq, q, p.head_dim, p.n_q_heads, total_tokens) ||
        !make_rows_tmap(&tk, k, p.head_dim, p.n_kv_heads, total_tokens) ||
        !make_rows_tmap(&tv, v, p.head_dim, p.n_kv_heads, total_tokens) ||
        !make_rows_tmap(&tkp, k_pages, p.head_dim, p.n_kv_heads, pool_rows, 16) ||
        !make_rows_tmap(&tvp, v_pages, p.head_dim, p.n_kv_heads, pool_rows, 16))
        return cudaErrorInvalidValue;
    AttnTcArgs a{};
    a.cu = cu_seqlens;
    a.out = static_cast<uint16_t *>(out);
    a.n_seg = batch;
    a.total = total_tokens;
    a.hq = p.n_q_heads;
    a.scale_log2 = scale * kLog2e;
    a.page_table = page_table;
    a.k_pages = static_cast<uint16_t *>(k_pages);
    a.v_pages = static_cast<uint16_t *>(v_pages);
    a.hkv = p.n_kv_heads;
    a.max_pages = p.max_pages_per_seq;
    a.num_pages = p.num_pages;
    a.page_size = p.page_size;
    a.n_past = n_past;
    a.early = (p.abi_version >= 2 && p.stable_metadata >= 1) ? 1 : 0;
    unsigned int *status = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status);
    if (e != cudaSuccess) return e;
    // a request holds at most max_pages_per_seq * page_size rows
    const long long max_len = (long long)p.max_pages_per_seq * p.page_size;
    const long long qtiles = (max_len + 127) / 128;
    if (qtiles > 65535 || batch > 65535) return cudaErrorInvalidValue;
    const dim3 grid(p.n_q_heads, batch, (unsigned)qtiles);
    // the chunked form keeps up to 256 cached page ids in 1 KiB more
    const uint32_t smem = AttnTcLayout<128>::kSmem + (n_past ? 1024u : 0u);
    auto launch = [&](auto kernel) -> cudaError_t {
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   (int)cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        // a programmatic dependent of the kernel before it on the stream:
        // its CTAs are scheduled as that kernel's last CTAs retire, and wait
        // for it (griddepcontrol.wait) before they read anything
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, tkp, tvp, a, status);
    };
    const bool group2 = p.n_q_heads == 2 * p.n_kv_heads;
    if (n_past)
        e = group2 ? launch(prefill_tc_kernel<2, true>) : launch(prefill_tc_kernel<1, true>);
    else
        e = group2 ? launch(prefill_tc_kernel<2, false>) : launch(prefill_tc_kernel<1, false>);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

unsigned int status_read_clear_prefill(cudaStream_t stream, cudaError_t *err) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status, sizeof v, 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && v) e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (err) *err = e;
    return v;
}

}  // namespace qa

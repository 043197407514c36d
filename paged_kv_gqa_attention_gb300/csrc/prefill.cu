// Ragged causal prefill: the KV page write and the causal attention.
//
// Page write (qwenasr.cpp ARCHITECTURE.md, "Qwen3 Thinker decoder": prefill
// rewinds the cache and writes the fresh K/V of the whole prompt span at
// [n_past, n_past + T) with n_past = 0): row i of request r is copied bit for
// bit to slot i % 16 of page page_table[r][i / 16], for K and V.
//
// Attention: row i of request r attends over rows j <= i of the same request
// (same section: attend over [0, n_past + T)), GQA group h / 2, from the
// packed k and v, on the tensor cores (attn_tc.cuh): one CTA per (128-row
// query tile, query head, request) with causal key tiles 0..tile; the two
// query heads of a KV head are adjacent in launch order, so their K/V tiles
// come from L2 the second time.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "qa_internal.h"
#include "attn_tc.cuh"
#include "tmap.h"

namespace qa {
namespace {

__device__ unsigned int g_status;

struct PageWriteArgs {
    const uint4 *k, *v;  // [T][row_chunks] 16-byte chunks
    const int32_t *cu;
    const int32_t *page_table;
    uint4 *k_pages, *v_pages;
    int batch, total, max_pages, num_pages, page_size, row_chunks;
};

// One CTA per packed row; thread c copies 16-byte chunk c of the row's K and
// V (row_chunks = Hkv * D * 2 / 16 chunks).
__global__ void page_write_kernel(const PageWriteArgs a) {
    const int t = blockIdx.x;
    int lo = 0, hi = a.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int r0 = a.cu[lo], r1 = a.cu[lo + 1];
    if (!(0 <= r0 && r0 <= t && t < r1 && r1 <= a.total) || a.cu[a.batch] != a.total) {
        if (threadIdx.x == 0) atomicOr(&g_status, QA_DEVICE_BAD_SEGMENTS);
        return;
    }
    const int i = t - r0;
    if (i >= a.max_pages * a.page_size) {
        if (threadIdx.x == 0) atomicOr(&g_status, QA_DEVICE_BAD_LENGTH);
        return;
    }
    const int page = a.page_table[(size_t)lo * a.max_pages + i / a.page_size];
    if (page < 0 || page >= a.num_pages) {
        if (threadIdx.x == 0) atomicOr(&g_status, QA_DEVICE_BAD_PAGE);
        return;
    }
    const size_t dst = ((size_t)page * a.page_size + i % a.page_size) * a.row_chunks;
    const size_t src = (size_t)t * a.row_chunks;
    for (int c = threadIdx.x; c < a.row_chunks; c += blockDim.x) {
        a.k_pages[dst + c] = a.k[src + c];
        a.v_pages[dst + c] = a.v[src + c];
    }
}

}  // namespace

cudaError_t launch_page_write(const void *k, const void *v, const int32_t *cu_seqlens, int batch,
                              int total_tokens, const int32_t *page_table, void *k_pages,
                              void *v_pages, const qa_attn_params &p, cudaStream_t stream) {
    if (total_tokens == 0) return cudaSuccess;
    PageWriteArgs a;
    a.k = static_cast<const uint4 *>(k);
    a.v = static_cast<const uint4 *>(v);
    a.cu = cu_seqlens;
    a.page_table = page_table;
    a.k_pages = static_cast<uint4 *>(k_pages);
    a.v_pages = static_cast<uint4 *>(v_pages);
    a.batch = batch;
    a.total = total_tokens;
    a.max_pages = p.max_pages_per_seq;
    a.num_pages = p.num_pages;
    a.page_size = p.page_size;
    a.row_chunks = p.n_kv_heads * p.head_dim * 2 / 16;
    const int threads = a.row_chunks < 128 ? ((a.row_chunks + 31) / 32) * 32 : 128;
    page_write_kernel<<<total_tokens, threads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                           int batch, int total_tokens, void *out, const qa_attn_params &p,
                           float scale, cudaStream_t stream) {
    if (total_tokens == 0) return cudaSuccess;
    if (batch > 65535) return cudaErrorInvalidValue;
    CUtensorMap tq, tk, tv;
    if (!make_rows_tmap(&tq, q, p.head_dim, p.n_q_heads, total_tokens) ||
        !make_rows_tmap(&tk, k, p.head_dim, p.n_kv_heads, total_tokens) ||
        !make_rows_tmap(&tv, v, p.head_dim, p.n_kv_heads, total_tokens))
        return cudaErrorInvalidValue;
    AttnTcArgs a;
    a.cu = cu_seqlens;
    a.out = static_cast<uint16_t *>(out);
    a.n_seg = batch;
    a.total = total_tokens;
    a.hq = p.n_q_heads;
    a.scale_log2 = scale * kLog2e;
    unsigned int *status = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status);
    if (e != cudaSuccess) return e;
    // a request holds at most max_pages_per_seq * page_size rows
    const long long max_len = (long long)p.max_pages_per_seq * p.page_size;
    const long long qtiles = (max_len + 127) / 128;
    if (qtiles > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (qtiles > 65535 || batch > 65535) return cudaErrorInvalidValue;
    const dim3 grid(p.n_q_heads, batch, (unsigned)qtiles);
    constexpr uint32_t smem = AttnTcLayout<128>::kSmem;
    if (p.n_q_heads == 2 * p.n_kv_heads) {
        e = cudaFuncSetAttribute(attn_tc_kernel<128, 2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attn_tc_kernel<128, 2, true><<<grid, 128, smem, stream>>>(tq, tk, tv, a, status);
    } else {
        e = cudaFuncSetAttribute(attn_tc_kernel<128, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attn_tc_kernel<128, 1, true><<<grid, 128, smem, stream>>>(tq, tk, tv, a, status);
    }
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

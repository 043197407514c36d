// Decode KV append: per-head QK-norm, NEOX RoPE and the page write of the new
// token, one launch for the whole batch.
//
// qwenasr.cpp ARCHITECTURE.md, "Qwen3 Thinker decoder": per layer, q and k
// get a per-head RMSNorm (RMS over head_dim, then a [head_dim] gain) and then
// a 1D NEOX RoPE with freq_base 1e6 ("Attention and RoPE": rotate-half
// layout); decode appends the new token at position cur_len and attends over
// [0, cur_len + 1).  Here cur_len = seq_lens[b] - 1 (seq_lens count the new
// token, as qa_decode_attn reads them).
//
// One CTA per request, one warp per head vector (the n_q_heads query heads,
// then the n_kv_heads key heads).  Lane l holds dims {2l, 2l+1} of the first
// half and {64+2l, 64+2l+1} of the second, so each lane owns the two rotation
// pairs (2l, 64+2l) and (2l+1, 64+2l+1) and every load and store is one
// coalesced 128-byte row segment.  In fp32: the mean of squares (warp sum),
// 1/sqrt(ms + eps), the gain, the rotation.  The angle cur * theta^(-2i/D)
// is carried as an exact fp32 sum and reduced modulo 2 pi by Cody-Waite
// (sincos_pos_freq; the per-pair frequencies are computed on the host in
// fp64 and passed as fp32 hi + lo parts), so large positions keep full fp32
// accuracy without fp64 arithmetic.  Results are rounded to bf16 (nearest
// even).  The V rows are copied unchanged by the first threads.
//
// The kernel waits on griddepcontrol before reading its inputs and lets its
// dependents launch at once, so the decode kernel that follows on the stream
// can be resident before the append ends (it waits for the append's
// completion before it reads anything).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "qa_internal.h"

namespace qa {
namespace {

__device__ unsigned int g_status;

constexpr int kD = 128;
constexpr int kPS = 16;
constexpr int kHalfWords = kD / 4;  // 32-bit words (bf16 pairs) in half a head vector

struct AppendArgs {
    const uint32_t *q, *k;  // [B][H][D] bf16, as bf16 pairs
    const uint4 *v;         // [B][Hkv][D] bf16, as 16-byte chunks
    const float2 *q_gain, *k_gain;
    const int32_t *page_table, *seq_lens;
    uint32_t *q_out, *k_pages;  // pools as bf16 pairs
    uint4 *v_pages;
    int hq, hkv, max_pages, num_pages;
    float eps;
    // theta^(-2i/D), computed on the host in fp64, as fp32 hi + lo parts
    float freq_hi[kD / 2], freq_lo[kD / 2];
};

__global__ void __launch_bounds__(1024) append_kernel(const __grid_constant__ AppendArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int len = a.seq_lens[b];
    if (len < 1 || len > a.max_pages * kPS) {
        if (threadIdx.x == 0) atomicOr(&g_status, QA_DEVICE_BAD_LENGTH);
        return;
    }
    const int cur = len - 1;
    const int page = a.page_table[(size_t)b * a.max_pages + cur / kPS];
    if (page < 0 || page >= a.num_pages) {
        if (threadIdx.x == 0) atomicOr(&g_status, QA_DEVICE_BAD_PAGE);
        return;
    }
    const size_t slot_row = (size_t)page * kPS + cur % kPS;  // row of the pool, [Hkv][D] per row

    // V: copied unchanged (Hkv * D * 2 bytes = Hkv * 16 chunks)
    const int v_chunks = a.hkv * (kD / 8);
    if ((int)threadIdx.x < v_chunks)
        a.v_pages[slot_row * v_chunks + threadIdx.x] = a.v[(size_t)b * v_chunks + threadIdx.x];

    if (warp >= a.hq + a.hkv) return;
    const bool is_q = warp < a.hq;
    const uint32_t *src = is_q ? a.q + ((size_t)b * a.hq + warp) * (kD / 2)
                               : a.k + ((size_t)b * a.hkv + (warp - a.hq)) * (kD / 2);
    const uint32_t w0 = src[lane], w1 = src[kHalfWords + lane];
    const float x0 = bf16lo(w0), x1 = bf16hi(w0);  // dims 2l, 2l+1
    const float y0 = bf16lo(w1), y1 = bf16hi(w1);  // dims 64+2l, 64+2l+1
    const float ss = warp_sum(x0 * x0 + x1 * x1 + y0 * y0 + y1 * y1);
    const float r = 1.0f / sqrtf(ss * (1.0f / kD) + a.eps);
    const float2 *gain = is_q ? a.q_gain : a.k_gain;
    const float2 g0 = gain[lane], g1 = gain[kHalfWords + lane];
    const float n0 = x0 * r * g0.x, n1 = x1 * r * g0.y;
    const float m0 = y0 * r * g1.x, m1 = y1 * r * g1.y;

    // angles of pairs 2l and 2l+1
    float s0, c0, s1, c1;
    sincos_pos_freq(cur, a.freq_hi[2 * lane], a.freq_lo[2 * lane], &s0, &c0);
    sincos_pos_freq(cur, a.freq_hi[2 * lane + 1], a.freq_lo[2 * lane + 1], &s1, &c1);
    const float z0 = n0 * c0 - m0 * s0, z1 = n1 * c1 - m1 * s1;  // first half
    const float u0 = n0 * s0 + m0 * c0, u1 = n1 * s1 + m1 * c1;  // second half
    uint32_t *dst = is_q ? a.q_out + ((size_t)b * a.hq + warp) * (kD / 2)
                         : a.k_pages + (slot_row * a.hkv + (warp - a.hq)) * (kD / 2);
    dst[lane] = pack_bf16x2(z0, z1);
    dst[kHalfWords + lane] = pack_bf16x2(u0, u1);
}

}  // namespace

cudaError_t launch_append(const void *q, const void *k, const void *v, const float *q_gain, const float *k_gain,
                          float rms_eps, float rope_theta, const int32_t *page_table, const int32_t *seq_lens,
                          int batch, void *k_pages, void *v_pages, void *q_out, const qa_attn_params &p,
                          cudaStream_t stream) {
    AppendArgs a;
    a.q = static_cast<const uint32_t *>(q);
    a.k = static_cast<const uint32_t *>(k);
    a.v = static_cast<const uint4 *>(v);
    a.q_gain = reinterpret_cast<const float2 *>(q_gain);
    a.k_gain = reinterpret_cast<const float2 *>(k_gain);
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.q_out = static_cast<uint32_t *>(q_out);
    a.k_pages = static_cast<uint32_t *>(k_pages);
    a.v_pages = static_cast<uint4 *>(v_pages);
    a.hq = p.n_q_heads;
    a.hkv = p.n_kv_heads;
    a.max_pages = p.max_pages_per_seq;
    a.num_pages = p.num_pages;
    a.eps = rms_eps;
    for (int i = 0; i < kD / 2; ++i) {
        const double f = pow((double)rope_theta, -2.0 * i / kD);
        a.freq_hi[i] = (float)f;
        a.freq_lo[i] = (float)(f - (double)a.freq_hi[i]);
    }

    const int warps = p.n_q_heads + p.n_kv_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)batch);
    cfg.blockDim = dim3((unsigned)(warps * 32));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_kernel, a);
}

unsigned int status_read_clear_append(cudaStream_t stream, cudaError_t *err) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status, sizeof v, 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && v) e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (err) *err = e;
    return v;
}

}  // namespace qa

// The AuT encoder layer around the window attention (qwenasr.cpp
// ARCHITECTURE.md, "Windowed audio tower": a pre-norm Whisper-style
// transformer layer, LayerNorm with bias, bias on q / k / v / output, gelu
// MLP; "GGUF layout": attn_norm, attn_q / attn_k / attn_v / attn_output,
// ffn_norm, ffn_up / ffn_down, each with weight and bias):
//
//   a = LN1(x);  q|k|v = a Wqkv^T + bqkv;  o = window attention(q, k, v)
//   h = x + (o Wo^T + bo)
//   f = gelu(LN2(h) W1^T + b1);  y = h + (f W2^T + b2)
//
// Seven launches on one stream, each a programmatic dependent of the one
// before: LayerNorm, the fused q|k|v projection (one [T][3 d] buffer), the
// window attention reading q, k and v straight out of that buffer (row
// stride 3 d), the output projection with bias and residual fused in its
// epilogue, LayerNorm, fc1 with bias and gelu fused, fc2 with bias and
// residual fused.  Every intermediate is bf16 (the operator boundaries).
// The window attention claims its jobs from a counter in the workspace,
// which the first LayerNorm zeroes.
//
// layer_norm_kernel: one warp per token row; lane l holds 4-element chunks
// l, l + 32, ... of the row (coalesced 8-byte loads), mean and biased
// variance by warp sums in fp32, y = (x - mean) / sqrt(var + eps) * g + b
// rounded to bf16.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "qa_internal.h"

namespace qa {
namespace {

constexpr int kLnMaxChunks = 16;  // d_model up to 16 * 128 = 2048

// CH: 4-element chunks per lane (d = 128 CH), a compile-time count so the
// row stays in 4 CH registers per lane (a short kernel that many warps of an
// SM run at once: that is what keeps enough loads in flight).
template <int CH>
__global__ void __launch_bounds__(256) layer_norm_kernel(const uint16_t *x, int T, const uint16_t *g,
                                                         const uint16_t *b, float eps, uint16_t *y, int *zero2) {
    constexpr int d = 128 * CH;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (zero2 && blockIdx.x == 0 && threadIdx.x < 2) zero2[threadIdx.x] = 0;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const uint2 *xr = reinterpret_cast<const uint2 *>(x + (size_t)t * d);
    uint2 w[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) w[c] = xr[c * 32 + lane];
    float v[CH][4];
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        v[c][0] = bf16lo(w[c].x), v[c][1] = bf16hi(w[c].x), v[c][2] = bf16lo(w[c].y), v[c][3] = bf16hi(w[c].y);
        s += (v[c][0] + v[c][1]) + (v[c][2] + v[c][3]);
    }
    const float mean = warp_sum(s) * (1.0f / d);
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float u = v[c][j] - mean;
            ss = fmaf(u, u, ss);
        }
    const float inv = rsqrtf(warp_sum(ss) * (1.0f / d) + eps);
    const uint2 *gr = reinterpret_cast<const uint2 *>(g);
    const uint2 *br = reinterpret_cast<const uint2 *>(b);
    uint2 *yr = reinterpret_cast<uint2 *>(y + (size_t)t * d);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const uint2 gw = gr[c * 32 + lane], bw = br[c * 32 + lane];
        const float o0 = fmaf((v[c][0] - mean) * inv, bf16lo(gw.x), bf16lo(bw.x));
        const float o1 = fmaf((v[c][1] - mean) * inv, bf16hi(gw.x), bf16hi(bw.x));
        const float o2 = fmaf((v[c][2] - mean) * inv, bf16lo(gw.y), bf16lo(bw.y));
        const float o3 = fmaf((v[c][3] - mean) * inv, bf16hi(gw.y), bf16hi(bw.y));
        yr[c * 32 + lane] = make_uint2(pack_bf16x2(o0, o1), pack_bf16x2(o2, o3));
    }
}

template <int CH>
cudaError_t launch_ln(const void *x, int T, const void *g, const void *b, float eps, void *y, cudaStream_t stream,
                      int *zero2) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((T + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, layer_norm_kernel<CH>, static_cast<const uint16_t *>(x), T,
                              static_cast<const uint16_t *>(g), static_cast<const uint16_t *>(b), eps,
                              static_cast<uint16_t *>(y), zero2);
}

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

}  // namespace

bool layer_norm_supported(int d) { return d >= 128 && d % 128 == 0 && d / 128 <= kLnMaxChunks; }

cudaError_t launch_layer_norm(const void *x, int T, int d, const void *g, const void *b, float eps, void *y,
                              cudaStream_t stream, int *zero2) {
    if (T == 0) return cudaSuccess;
    cudaError_t e;
    switch (d / 128) {
        case 1: e = launch_ln<1>(x, T, g, b, eps, y, stream, zero2); break;
        case 2: e = launch_ln<2>(x, T, g, b, eps, y, stream, zero2); break;
        case 3: e = launch_ln<3>(x, T, g, b, eps, y, stream, zero2); break;
        case 4: e = launch_ln<4>(x, T, g, b, eps, y, stream, zero2); break;
        case 5: e = launch_ln<5>(x, T, g, b, eps, y, stream, zero2); break;
        case 6: e = launch_ln<6>(x, T, g, b, eps, y, stream, zero2); break;
        case 7: e = launch_ln<7>(x, T, g, b, eps, y, stream, zero2); break;
        case 8: e = launch_ln<8>(x, T, g, b, eps, y, stream, zero2); break;
        case 9: e = launch_ln<9>(x, T, g, b, eps, y, stream, zero2); break;
        case 10: e = launch_ln<10>(x, T, g, b, eps, y, stream, zero2); break;
        case 11: e = launch_ln<11>(x, T, g, b, eps, y, stream, zero2); break;
        case 12: e = launch_ln<12>(x, T, g, b, eps, y, stream, zero2); break;
        case 13: e = launch_ln<13>(x, T, g, b, eps, y, stream, zero2); break;
        case 14: e = launch_ln<14>(x, T, g, b, eps, y, stream, zero2); break;
        case 15: e = launch_ln<15>(x, T, g, b, eps, y, stream, zero2); break;
        case 16: e = launch_ln<16>(x, T, g, b, eps, y, stream, zero2); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

EncoderWorkspace encoder_workspace_layout(long long T, int d, int d_ffn) {
    EncoderWorkspace w;
    w.ctr = 0;
    w.a = 256;
    w.qkv = w.a + align256((size_t)T * d * 2);
    w.o = w.qkv + align256((size_t)T * 3 * d * 2);
    w.h = w.o + align256((size_t)T * d * 2);
    w.f = w.h + align256((size_t)T * d * 2);
    w.total = w.f + align256((size_t)T * d_ffn * 2);
    return w;
}

cudaError_t launch_encoder_layer(const void *x, const int32_t *cu_windows, int n_windows, int T, int d, int H,
                                 int d_ffn, const qa_encoder_weights &w, float eps, void *workspace, void *out,
                                 const qa_attn_params &p, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const EncoderWorkspace L = encoder_workspace_layout(T, d, d_ffn);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *a = ws + L.a, *qkv = ws + L.qkv, *o = ws + L.o, *h = ws + L.h, *f = ws + L.f;
    int *job_ctr = reinterpret_cast<int *>(ws + L.ctr);
    const uint16_t *qkv16 = static_cast<const uint16_t *>(qkv);
    cudaError_t e;
    // attention block
    // the first LayerNorm also zeroes the window attention's job counter
    // (the workspace holds anything on entry)
    if ((e = launch_layer_norm(x, T, d, w.ln1_g, w.ln1_b, eps, a, stream, job_ctr)) != cudaSuccess) return e;
    if ((e = launch_gemm(a, d, T, d, w.w_qkv, 3 * d, w.b_qkv, 0, nullptr, 0, qkv, 3 * d, stream)) != cudaSuccess)
        return e;
    qa_attn_params pw = p;
    pw.n_q_heads = pw.n_kv_heads = H;
    pw.head_dim = d / H;
    if ((e = launch_window(qkv16, qkv16 + d, qkv16 + 2 * d, cu_windows, n_windows, T, o, pw,
                           1.0f / sqrtf((float)(d / H)), stream, 3LL * d, job_ctr)) != cudaSuccess)
        return e;
    if ((e = launch_gemm(o, d, T, d, w.w_o, d, w.b_o, 0, x, d, h, d, stream)) != cudaSuccess) return e;
    // MLP block
    if ((e = launch_layer_norm(h, T, d, w.ln2_g, w.ln2_b, eps, a, stream)) != cudaSuccess) return e;
    if ((e = launch_gemm(a, d, T, d, w.w_fc1, d_ffn, w.b_fc1, 1, nullptr, 0, f, d_ffn, stream)) != cudaSuccess)
        return e;
    return launch_gemm(f, d_ffn, T, d_ffn, w.w_fc2, d, w.b_fc2, 0, h, d, out, d, stream);
}

}  // namespace qa
